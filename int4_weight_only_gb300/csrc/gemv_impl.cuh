// gemv_impl.cuh - decode kernels (M <= 16) for the INT4 weight-only linear
// layer.  Each translation unit instantiates one family, so that adding a
// family leaves the others' generated code as it was:
//   gemv.cu         planner; W4A16 unsplit plans; W4A8 (one scale per row)
//   gemv_split.cu   W4A16 K-split plans
//   gemv_swiglu.cu  SWIGLU: gate|up row pairs, SiLU(gate) * up epilogue
//   gemv_grouped.cu GROUPED: one matrix per group of tokens (experts)
//   gemv_bf16p.cu   SB: bf16 scales and (8 - z) s offsets
//   gemv_w4a8g.cu   W4A8 with one scale per group of G columns
//   gemv_f32.cu     F32: fp32 partial outputs of a row-parallel shard
//   gemv_swiglu_q8.cu Q8: SWIGLU with INT8 outputs for the W4A8 GEMV
//
// W4A16 ("Lab 5: Gemma4 端到端推理优化", sections "INT4 线性量化" and
// "融合INT4反量化与矩阵乘"): y = x W_hat^T (+b) with W_hat = s (code - z),
// dequantized in registers next to the multiply, one pass over the packed
// weights.  W4A8 ("Jetson Orin AGX INT4 推理优化实践", sections
// "从 FP 线性层到 INT4 DP4A 的数学推导" and "DP4A 做了什么"):
// acc = sum (code - 8) q_x in int32, y = s_W s_x acc + b.
//
// Structure (both kernels): persistent CTAs of 8 consumer warps + 1
// producer warp, one or two CTAs per SM.  A unit of work is (block of R
// output rows, slice of the padded K), R in {16, 32, 64, 128}; units are dealt
// round-robin to the CTAs.  The producer streams 16 KB stages of packed
// weights (128/R TMA boxes of R rows x 128 bytes, 128-byte swizzle) into a
// 3-deep ring.  Each stage holds eight 16-row x 256-column boxes; consumer
// warp w takes row tile w % (R/16) and k-phase w / (R/16), i.e. exactly one
// such box per stage, and reads it with ldmatrix.  Partial sums of the
// k-phases are added in shared memory in a fixed order; K slices of a row
// block (split-K) are added by the last CTA to finish it, also in a fixed
// order, so results are deterministic.
//
// W4A16 inner product: each 32-bit ldmatrix word holds 8 codes of one row;
// one LOP3 per pair ORs the codes into the mantissa of fp16 1024.0 (both
// nibbles of a byte fit the 10-bit mantissa, as 1024 + c and 1024 + 16c),
// and one f16x2 subtraction of the row's 1024 + z (1024 + 16z) leaves
// (c - z) and 16 (c - z), small integers held exactly.  These words feed
// mma.sync m16n8k16 (fp16 inputs, fp32 accumulation) as the A operand (16
// weight rows), with the activations as the B operand (8 tokens per n-tile).
// The activations are converted to fp16 exactly: each token's slice is
// scaled by a power of two first (undone in the epilogue), odd columns also
// by 1/16.  The order of k inside a 32-column chunk is permuted identically
// on both operands, so no data shuffles are needed.  Every product is exact
// in fp32; the MMAs of one group's run of columns accumulate into a fresh
// register set, which is then scaled by the group's s and added to the
// running sums.

// Launch: programmatic dependent launch.  Before waiting for the previous
// kernel on the stream, each CTA reads only constant inputs: the producer
// prefetches the first stages of its first unit into L2, the consumers load
// their first scales and their bias.  x, the workspace, y and every
// shared-memory copy come after griddepcontrol.wait.
#pragma once

#include "w4_device.cuh"
#include "w4_internal.h"

#include <algorithm>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

namespace w4 {
namespace {

constexpr int CW = kGemvConsumerWarps;
constexpr int NCT = CW * 32;
constexpr int NS = kGemvStages;
constexpr int STAGE_BYTES = kGemvStageBytes;

// the producer's mark in the first segment's (unused) fourth sum on the fp16
// path, until the consumers' staging writes 0 there
constexpr uint32_t kXsegSentinel = 0xFFFFFFFFu;

struct SmemCtl {
    uint64_t full[NS];
    uint64_t empty[NS];
    int abort;
    int last;
    int sumq[16];          // W4A8: sum of q_x over the slice, per token; W4A16
                           // with INT8 outputs: the CTA's max|y| per token (fp32 bits)
    uint64_t xfull;        // activation slice landed (TMA staging)
    uint64_t xempty;       // consumers released the activation buffer
    uint64_t listready;    // grouped: the (group, token tile) list is written
    int nact;              // grouped: number of items in it
    uint64_t cready;       // cluster split, rank 0: the other ranks' partials landed
    int gen;               // INT8 outputs: the call's generation (maxima buffer parity)
};
constexpr int kCtlBytes = 256;
static_assert(sizeof(SmemCtl) <= kCtlBytes, "control block");

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

__device__ __forceinline__ void grid_dep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1) : "memory");
}

// Producer: one thread streams every stage of every unit of this CTA.
// GROUPED: units are ((group, token tile) item, row block) in the order of
// the list the consumers build after the dependency wait; rows of group e
// start at e * N.
template <bool GROUPED = false>
__device__ void gemv_producer(const CUtensorMap* tm, uint8_t* wbuf, uint8_t* xbuf,
                              SmemCtl* ctl, const GemvArgs& a) {
    const int boxes = 128 / a.R;
    const int box_bytes = a.R * 128;
    const int kbytes = a.Kp / 2;
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int slot, int ks, int row) {
        const int kb0 = ks * (a.SKE / 2);
        const int nbox = min(boxes, (kbytes - kb0 + 127) / 128);   // boxes inside Kp
        mbar_arrive_expect_tx(&ctl->full[slot], nbox * box_bytes);
        for (int b = 0; b < nbox; ++b)
            tma_load_2d(wbuf + slot * STAGE_BYTES + b * box_bytes, tm, kb0 + b * 128, row,
                        &ctl->full[slot], pol);
    };
    // fp16 path with the activations read by the consumers: after a.xfirst
    // stages of the first unit the rest of the ring is held until the
    // consumers have staged their slice, so that their activation loads do
    // not queue behind every CTA's whole ring of weight copies.  Their
    // staging writes 0 into the unused fourth sum of the first segment; the
    // producer leaves a sentinel there first (the consumers start staging
    // only after the dependency wait and an activation load) and watches it.
    // A hint only: the watch gives up after about two microseconds, and the
    // word is never read by the arithmetic.
    int hold = GROUPED ? -1 : a.xfirst;
    volatile uint32_t* const xflag =
        reinterpret_cast<volatile uint32_t*>(xbuf + (size_t)a.M * a.XS) + 3;
    if (hold >= 0) *xflag = kXsegSentinel;
    // The weights are not written by the kernel before this one on the
    // stream, so while it may still be running the first unit's first a.pf
    // stages are prefetched into L2.  (Loading them into shared memory here
    // instead was measured slower: those copies compete with the activation
    // copy that follows the wait for the SM's bandwidth.)
    if (!GROUPED && (int)blockIdx.x < a.units) {
        int rb, s, ks0, ks1;
        unit_coords(blockIdx.x, a, rb, s, ks0, ks1);
        for (int ks = ks0; ks < min(ks1, ks0 + a.pf); ++ks)
            for (int b = 0; b < boxes; ++b) {
                const int kb = ks * (a.SKE / 2) + b * 128;
                if (kb < kbytes) tma_prefetch_l2_2d(tm, kb, rb * a.R);
            }
    }
    grid_dep_wait();
    int units = a.units;
    const int* glist = nullptr;
    if constexpr (GROUPED) {
        // which groups have tokens is known only after the wait
        if (!mbar_wait(&ctl->listready, 0, &ctl->abort, a.err)) return;   // nothing issued yet
        units = ctl->nact * a.NBg;
        glist = reinterpret_cast<const int*>(wbuf + a.list_off);
    }
    // GROUPED: each CTA takes a contiguous run of units, so that successive
    // units mostly share a group and its staged activations
    int u_beg = blockIdx.x, u_end = units, u_step = gridDim.x;
    if constexpr (GROUPED) {
        u_beg = (int)(((long long)units * blockIdx.x) / gridDim.x);
        u_end = (int)(((long long)units * (blockIdx.x + 1)) / gridDim.x);
        u_step = 1;
    }
    uint32_t it = 0, xi = 0;
    int pv0 = -1, pv1 = -1;
    bool ok = true;
    for (int u = u_beg; u < u_end && ok; u += u_step) {
        int rb, s, ks0, ks1, row;
        if constexpr (GROUPED) {
            const int gi = u / a.NBg;
            rb = u - gi * a.NBg;
            s = 0; ks0 = 0; ks1 = a.nst;
            row = (glist[gi] & 0xFFFF) * a.N + rb * a.R;
        } else {
            unit_coords(u, a, rb, s, ks0, ks1);
            row = rb * a.R;
        }
        if (a.xtma && (ks0 != pv0 || ks1 != pv1)) {
            // the activation slice goes out before this unit's weights
            if (xi > 0 && !mbar_wait(&ctl->xempty, (xi - 1) & 1, &ctl->abort, a.err)) {
                ok = false;
                break;
            }
            const int k0 = ks0 * a.SKE;
            const int ncol = min((ks1 - ks0) * a.SKE, a.K - k0);
            const uint32_t nbytes = ncol > 0 ? (uint32_t)ncol * 2u : 0u;
            mbar_arrive_expect_tx(&ctl->xfull, nbytes * (uint32_t)a.M);
            if (nbytes)
                for (int m = 0; m < a.M; ++m)
                    bulk_load(xbuf + (size_t)m * a.XS,
                              static_cast<const uint16_t*>(a.x) + (size_t)m * a.K + k0, nbytes,
                              &ctl->xfull);
            ++xi;
            pv0 = ks0;
            pv1 = ks1;
        }
        for (int ks = ks0; ks < ks1; ++ks, ++it) {
            const int slot = it % NS;
            if (hold >= 0 && it == (uint32_t)hold) {
                for (int i = 0; i < 64 && *xflag == kXsegSentinel; ++i) __nanosleep(16);
                hold = -1;
            }
            if (it >= (uint32_t)NS &&
                !mbar_wait(&ctl->empty[slot], ((it / NS) & 1) ^ 1, &ctl->abort, a.err)) {
                ok = false;
                break;
            }
            issue(slot, ks, row);
        }
    }
    if (!ok || ctl->abort) {
        // A wait gave up: let the copies already issued land before exiting.
        const uint32_t first = it > (uint32_t)NS ? it - NS : 0;
        for (uint32_t j = first; j < it; ++j)
            mbar_wait_drain(&ctl->full[j % NS], (j / NS) & 1, a.err);
        if (xi > 0) mbar_wait_drain(&ctl->xfull, (xi - 1) & 1, a.err);
    }
}

// Activations of one unit in shared memory: bf16 rows of columns [k0,
// k0+nk) as they are in x (nk a multiple of 256), columns >= K zero (the
// padded weights there are zero, but stale shared memory could hold NaNs).
// FROM_SMEM: the producer's copy of the first ncol columns has landed (K a
// multiple of 8), only the zero tail is written; otherwise the threads copy
// the slice from global memory.
template <bool FROM_SMEM>
__device__ __forceinline__ void stage_x_bf16(uint8_t* xbuf, const uint16_t* x, int M, int K,
                                             int XS, int k0, int nk, int tid) {
    const int nblk = nk >> 3;
    const int ncol = min(nk, K - k0);                  // columns inside x
    const int b0 = FROM_SMEM ? ncol >> 3 : 0;          // first block written here
    const int nb = nblk - b0, items = M * nb;
    const bool vec = (K & 7) == 0;
    for (int i = tid; i < items; i += NCT) {
        const int m = i / nb, b = b0 + (i - m * nb);
        const int k = k0 + b * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (!FROM_SMEM) {
            const uint16_t* src = x + (size_t)m * K + k;
            if (vec && k + 8 <= K) {
                v = __ldg(reinterpret_cast<const uint4*>(src));
            } else if (k < K) {
                uint16_t e[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) e[j] = (k + j < K) ? __ldg(src + j) : (uint16_t)0;
                v = make_uint4((uint32_t)e[0] | ((uint32_t)e[1] << 16), (uint32_t)e[2] | ((uint32_t)e[3] << 16),
                               (uint32_t)e[4] | ((uint32_t)e[5] << 16), (uint32_t)e[6] | ((uint32_t)e[7] << 16));
            }
        }
        *reinterpret_cast<uint4*>(xbuf + (size_t)m * XS + b * 16) = v;
    }
}

// F16 path: activations of one unit into shared memory as fp16, columns
// [k0, k0+nk).
// nk is a multiple of 256, so the slice is a whole number of segments of
// CPG*32 columns (one group's share of a box, BLK = CPG*4 blocks of 8
// columns).  An item is one (token, segment); L neighbouring lanes take it,
// lane l converting the segment's blocks l, l+L, ... (BPL = BLK/L of them),
// and log2(L) shuffle steps combine the segment.  L is chosen on the fly: the
// fewest passes of the 256 threads over the items with at most 8 blocks a
// lane (4 in the 96-register instances), then the most lanes that keep that
// number of passes.  Each lane first
// loads all its blocks into registers and only then uses them, so a pass costs
// one load latency, not one per block.  bf16 values are exactly
// representable in fp16 once a segment is scaled by a power of two 2^-e that
// puts its max|x| in [2^14, 2^15); odd columns of every 8-column block are
// further divided by 16 (exact) to match the 1024 + 16c weights of
// nibbles_to_f16x2_biased, and each block is stored in the order
// (0,4,1,5,2,6,3,7).  Columns >= K are zero.  Per segment and token,
// xseg[4 * (segment * M + token) + {0, 1, 2}] holds u = 2^e,
// u * (1024 E + 64 O) and u * (E + O), with E and O the sums of the scaled
// x over even and odd columns (each lane sums its blocks in order, then the
// L lanes are combined by xor-1, xor-2, ... shuffles): the MMA of the
// segment then equals u^-1 * (sum (c - z) x) + C0 + z * C1.
// FROM_SMEM: the raw bf16 slice was already copied into xbuf (row m at
// m * XS, natural order) and is converted in place; columns >= K hold stale
// data there and are replaced by zeros.
template <int CPG, int L, bool FROM_SMEM>
__device__ __forceinline__ void stage_x_f16_lanes(uint8_t* xbuf, float* xseg, const uint16_t* x,
                                                  int M, int K, int XS, int k0, int nseg,
                                                  int tid) {
    constexpr int BLK = CPG * 4, BPL = BLK / L;
    static_assert(BPL >= 1 && BPL <= 8 && L <= 32, "lanes per segment");
    const int items = M * nseg * L;
    const bool vec = (K & 7) == 0;
    const int lane = tid & 31;
    // whole warps iterate together so that every shuffle sees all 32 lanes;
    // items is a multiple of L, so a segment's lanes are all on or all off
    for (int base = tid - lane; base < items; base += NCT) {
        const int idx = base + lane;
        const bool on = idx < items;
        const int l = idx & (L - 1), ts = on ? idx / L : 0;
        const int m = ts / nseg, sg = ts - m * nseg;
        uint32_t q[BPL][4];
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            const int b = sg * BLK + l + L * i;          // block within the slice
            const int k = k0 + b * 8;
            const uint16_t* src = x + (size_t)m * K + k;
            if (!on) {
                q[i][0] = q[i][1] = q[i][2] = q[i][3] = 0u;
            } else if (FROM_SMEM) {
                if (k < K) {
                    const uint4 v = *reinterpret_cast<const uint4*>(xbuf + (size_t)m * XS + b * 16);
                    q[i][0] = v.x; q[i][1] = v.y; q[i][2] = v.z; q[i][3] = v.w;
                } else {
                    q[i][0] = q[i][1] = q[i][2] = q[i][3] = 0u;
                }
            } else if (vec && k + 8 <= K) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
                q[i][0] = v.x; q[i][1] = v.y; q[i][2] = v.z; q[i][3] = v.w;
            } else {
                uint16_t e[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) e[j] = (k + j < K) ? __ldg(src + j) : (uint16_t)0;
#pragma unroll
                for (int j = 0; j < 4; ++j) q[i][j] = (uint32_t)e[2 * j] | ((uint32_t)e[2 * j + 1] << 16);
            }
        }
        unsigned mx = 0;                      // bits of max|x| (non-negative floats order as ints)
#pragma unroll
        for (int i = 0; i < BPL; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                mx = max(mx, max((q[i][j] << 16) & 0x7FFFFFFFu, q[i][j] & 0x7FFF0000u));
#pragma unroll
        for (int o = 1; o < L; o <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const int E = (int)(mx >> 23) - 127;
        const int e = mx == 0 ? 0 : max(E - 14, -100);
        const float sc = __int_as_float((127 - e) << 23);
        float se = 0.f, so = 0.f;
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[2 * j] = __uint_as_float(q[i][j] << 16) * sc;
                v[2 * j + 1] = __uint_as_float(q[i][j] & 0xFFFF0000u) * sc;
            }
            se += (v[0] + v[2]) + (v[4] + v[6]);
            so += (v[1] + v[3]) + (v[5] + v[7]);
            const float s16 = 0.0625f;
            const int b = sg * BLK + l + L * i;
            if (on)
                *reinterpret_cast<uint4*>(xbuf + (size_t)m * XS + b * 16) =
                    make_uint4(pack_f16x2(v[0], v[4]), pack_f16x2(v[1] * s16, v[5] * s16),
                               pack_f16x2(v[2], v[6]), pack_f16x2(v[3] * s16, v[7] * s16));
        }
#pragma unroll
        for (int o = 1; o < L; o <<= 1) {
            se += __shfl_xor_sync(0xffffffffu, se, o);
            so += __shfl_xor_sync(0xffffffffu, so, o);
        }
        if (on && l == 0) {
            const float u = __int_as_float((127 + e) << 23);
            *reinterpret_cast<float4*>(xseg + 4 * (sg * M + m)) =
                make_float4(u, u * fmaf(1024.f, se, 64.f * so), u * (se + so), 0.f);
        }
    }
}

// MAXBPL: at most this many blocks (4 registers each) a lane, so that the
// staging fits the register budget of the kernel instance it is inlined in.
template <int CPG, bool FROM_SMEM, int MAXBPL>
__device__ __forceinline__ void stage_x_f16(uint8_t* xbuf, float* xseg, const uint16_t* x, int M,
                                            int K, int XS, int k0, int nk, int tid) {
    constexpr int BLK = CPG * 4;
    constexpr int LMIN = BLK > MAXBPL ? BLK / MAXBPL : 1;
    const int nseg = nk / (CPG * 32);
    const int items = M * nseg;
    const int passes = (items * LMIN + NCT - 1) / NCT;
    int L = LMIN;
    while (L * 2 <= BLK && L * 2 <= 32 && (items * L * 2 + NCT - 1) / NCT <= passes) L *= 2;
    switch (L) {
#define W4_STAGE_CASE(LL)                                                                      \
    case LL:                                                                                   \
        if constexpr (LL >= LMIN && LL <= BLK && LL <= 32)                                     \
            stage_x_f16_lanes<CPG, LL, FROM_SMEM>(xbuf, xseg, x, M, K, XS, k0, nseg, tid);     \
        break;
        W4_STAGE_CASE(1) W4_STAGE_CASE(2) W4_STAGE_CASE(4) W4_STAGE_CASE(8) W4_STAGE_CASE(16)
        W4_STAGE_CASE(32)
#undef W4_STAGE_CASE
        default: break;
    }
}

// INT8 activations of one unit, order (0,2,4,6 | 1,3,5,7) per 8-column
// block to match the byte lanes of (v & 0x0F0F0F0F) and ((v >> 4) & ...);
// also accumulates sum(q_x) over the slice per token into ctl->sumq (which
// the caller zeroed).
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

// Shared layout of one CTA; identical for both kernels.
struct Smem {
    uint8_t* wbuf;
    SmemCtl* ctl;
    float* red;
    uint8_t* xbuf;
    float* xseg;      // F16 path: per-segment sums of x, after M * XS bytes of xbuf
};

template <bool GROUPED = false>
__device__ __forceinline__ Smem gemv_init(const CUtensorMap* tm, const GemvArgs& a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = align1024(smem_raw);
    Smem sm;
    sm.wbuf = base;
    sm.ctl = reinterpret_cast<SmemCtl*>(base + NS * STAGE_BYTES);
    sm.red = reinterpret_cast<float*>(base + NS * STAGE_BYTES + kCtlBytes);
    sm.xbuf = base + NS * STAGE_BYTES + kCtlBytes + a.red;
    // the activation buffer holds M rows, or the per-group bound when grouped
    // (a.M is then the total row count of all groups)
    sm.xseg = reinterpret_cast<float*>(sm.xbuf + (size_t)(GROUPED ? a.gmax : a.M) * a.XS);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&sm.ctl->full[i], 1);
            mbar_init(&sm.ctl->empty[i], CW);
        }
        mbar_init(&sm.ctl->xfull, 1);
        mbar_init(&sm.ctl->xempty, 1);
        if constexpr (GROUPED) mbar_init(&sm.ctl->listready, 1);
        if (a.csplit) mbar_init(&sm.ctl->cready, a.S - 1);
        sm.ctl->abort = 0;
        sm.ctl->last = 0;
        for (int i = 0; i < 16; ++i) sm.ctl->sumq[i] = 0;

        fence_mbar_init();
    }
    if (threadIdx.x == NCT) tma_prefetch_desc(tm);
    grid_dep_launch();
    __syncthreads();
    // cluster split: every rank's barriers are initialized before any remote
    // arrival (all threads of every CTA of the cluster pass here once)
    if (a.csplit) cluster_sync();
    return sm;
}

// SiLU(gate) * up in fp32 (SiLU(v) = v * sigmoid(v)); __expf overflows to
// inf for very negative v and the reciprocal of inf is 0, the limit.  The
// correctly rounded reciprocal intrinsic keeps the epilogue branch-free.
__device__ __forceinline__ float swiglu(float gate, float up) {
    return gate * __frcp_rn(1.f + __expf(-gate)) * up;
}

// Sum of S split partials p[0], p[stride], ..., added in split order.  The
// loads of up to CH splits are issued before any add, so the last CTA of a
// row block waits for one round trip per CH splits, not one per split.
template <typename T, int CH = 8>
__device__ __forceinline__ T sum_splits(const T* p, size_t stride, int S) {
    T v = 0;
    for (int q = 0; q < S; q += CH) {
        T t[CH];
#pragma unroll
        for (int i = 0; i < CH; ++i)
            if (q + i < S) t[i] = ld_cg(p + (size_t)(q + i) * stride);
#pragma unroll
        for (int i = 0; i < CH; ++i)
            if (q + i < S) v += t[i];
    }
    return v;
}

// Split-K hand-off: after this CTA's partials are written, the last CTA of
// row block rb sees ctl->last set.  All consumer threads call it.  The CTA
// barrier orders every thread's partial stores before thread 0's ticket,
// whose acquire-release add at GPU scope publishes them to, and in the last
// CTA makes visible, the other splits' stores (no full fence per thread).
__device__ __forceinline__ bool split_k_arrive(const GemvArgs& a, SmemCtl* ctl, int rb) {
    named_bar_sync(1, NCT);
    if (threadIdx.x == 0) ctl->last = atom_add_acq_rel_gpu(&a.tickets[rb], 1) == a.S - 1;
    named_bar_sync(1, NCT);
    return ctl->last;
}

// The INT8 epilogue of the fused SwiGLU call ("Jetson Orin AGX INT4
// 推理优化实践", section 后续还能继续优化什么, item 2: the activation
// quantization folded into the op before the integer GEMV).
// q8_cta_max, called by all lanes of an epilogue warp per stored output: the
// max of |y| (bf16-rounded, as stored) over the lanes that hold the same
// token, then one shared-memory atomic max per token into ctl->sumq (|y| >= 0
// orders as an integer).
__device__ __forceinline__ void q8_cta_max(SmemCtl* ctl, float v, int t, int M, int lane,
                                           bool valid) {
    float m = valid ? fabsf(__uint_as_float((uint32_t)f32_to_bf16_bits(v) << 16)) : 0.f;
    // lanes with the same tig hold the same tokens: combine over gid
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
    if ((lane >> 2) == 0 && t < M && m > 0.f) atomicMax(&ctl->sumq[t], __float_as_int(m));
}

// Called by every consumer thread once its CTA has no units left.  The CTA
// adds its maxima with one atomic max per token on a.ymax[buffer], where the
// buffer is the parity of the call's generation a.gen[0] (so that a call
// never meets the previous call's maxima), then:
// * cooperative launch (a.coop, every CTA resident): a grid-wide barrier
//   (an acquire-release arrival count; the last CTA to arrive clears the
//   count and the other buffer, then releases the next generation, which
//   the others wait for with the usual bound), after which every CTA
//   quantizes its own share of y;
// * otherwise the CTA that takes the last ticket, which sees every CTA's y
//   and maxima, quantizes all of y.
// The rule is w4a8_quantize_act's: s_x = fp32(max|y| / 127), q = clip(rint(
// fp32(y / s_x)), -127, 127), columns F .. Fp-1 zero.
// IN: 16-byte loads in flight per thread in a pass.
template <int IN>
__device__ __forceinline__ void swiglu_q8_finish(const GemvArgs& a, SmemCtl* ctl, float* red,
                                                 int tid) {
    int* genp = a.done - 1;
    if (tid == 0) ctl->gen = ld_acquire_gpu(genp);      // this call's generation
    named_bar_sync(1, NCT);                  // the CTA's shared maxima are final
    const int g0 = ctl->gen;
    unsigned* ymax = a.ymax + 16 * (g0 & 1);
    if (tid < a.M && ctl->sumq[tid] != 0) atomicMax(ymax + tid, (unsigned)ctl->sumq[tid]);
    named_bar_sync(1, NCT);                  // this CTA's y stores and maxima are all issued
    const int F = a.N >> 1, nw = F >> 3, nwp = a.Fp >> 3;
    const int total = a.M * nwp;
    int w0 = 0, w1 = total;                  // this CTA's share of the (token, word) pairs
    if (a.coop) {
        if (tid == 0) {
            int ok = 1;
            if (atom_add_acq_rel_gpu(a.done, 1) == (int)gridDim.x - 1) {
                *a.done = 0;
                unsigned* other = a.ymax + 16 * ((g0 + 1) & 1);   // the previous call's
                for (int i = 0; i < 16; ++i) other[i] = 0u;
                st_release_gpu(genp, g0 + 1);
            } else {
                const long long t0 = clock64(), lim = wait_limit_of(a.err);
                while (ld_acquire_gpu(genp) == g0) {
                    if (clock64() - t0 > lim) {
                        atomicCAS(a.err, 0, W4_ERR_DEVICE_TIMEOUT);
                        ok = 0;
                        break;
                    }
                }
            }
            ctl->last = ok;
        }
        named_bar_sync(1, NCT);
        if (!ctl->last) return;
        w0 = (int)(((long long)total * blockIdx.x) / gridDim.x);
        w1 = (int)(((long long)total * (blockIdx.x + 1)) / gridDim.x);
    } else {
        if (tid == 0) ctl->last = atom_add_acq_rel_gpu(a.done, 1) == (int)gridDim.x - 1;
        named_bar_sync(1, NCT);
        if (!ctl->last) return;
    }
    if (tid < a.M) {
        const float mx = __uint_as_float(ld_cg_s32(reinterpret_cast<const int*>(ymax) + tid));
        const float sc = __fdiv_rn(mx, 127.0f);
        red[2 * tid] = sc;
        red[2 * tid + 1] = sc != 0.f ? __frcp_rn(sc) : 0.f;
        if (!a.coop || blockIdx.x == 0) a.sx_out[tid] = sc;
    }
    named_bar_sync(1, NCT);
    for (int base = w0 + tid; base < w1; base += IN * NCT) {
        uint4 v[IN];
#pragma unroll
        for (int i = 0; i < IN; ++i) {
            const int idx = base + i * NCT, m = idx / nwp, w = idx - m * nwp;
            v[i] = (idx < w1 && w < nw) ? ld_cg_v4(a.y + (size_t)m * F + 8 * w)
                                        : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < IN; ++i) {
            const int idx = base + i * NCT;
            if (idx >= w1) break;
            const int m = idx / nwp, w = idx - m * nwp;
            const uint32_t q[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            float f[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[2 * j] = __uint_as_float(q[j] << 16);
                f[2 * j + 1] = __uint_as_float(q[j] & 0xFFFF0000u);
            }
            *reinterpret_cast<uint2*>(a.qx + (size_t)m * a.Fp + 8 * w) =
                w < nw ? quant_s8x8(f, red[2 * m], red[2 * m + 1]) : make_uint2(0u, 0u);
        }
    }
    if (!a.coop) {
        named_bar_sync(1, NCT);
        if (tid < a.M) ymax[tid] = 0u;
        if (tid == 0) *a.done = 0;
    }
}

// SPLIT: the plan splits K (Sp > 1).  The two cases are separate kernels
// so that the split-K hand-off code does not take part in the register
// allocation and scheduling of the unsplit kernels' main loop (measured: it
// slowed that loop by ~4%).
// SWIGLU: the rows are gate/up pairs (16-row tiles: 8 gate rows, then the
// same 8 up rows) and y [M, N/2] = SiLU(gate) * up, SiLU(v) = v / (1 + e^-v).
// GROUPED: a grouped linear over E groups (experts): group e multiplies its
// own tokens, rows goff[e] .. goff[e+1] - 1 of x, by its own N x K matrix
// (rows e * N .. e * N + N - 1 of the stacked weights) into the same rows
// of y.  After the dependency wait every CTA lists the (group, token tile)
// items, tiles of at most gmax tokens, in group order (a block-wide prefix
// sum of the groups' tile counts), and takes a contiguous run of the
// (item, row block) units; a group whose offsets are invalid is left out
// and raises W4_ERR_GROUP_TOKENS.  Item = group | tile << 16.
// SB: bf16 parameters (a.scales_b, and for ASYM the offsets a.offs_b =
// bf16((8 - z) s) in place of zero points): w_hat = s (code - 8) + o, so the
// fix-up of a run is s (u tmp - C0 - 8 C1) + o C1.
// F32: fp32 outputs a.y32 without the bias (the partial sum of a row-
// parallel shard, added across shards and finished by w4a16_partial_finish).
// Q8 (with SWIGLU): the last CTA to finish also quantizes the whole output
// y [M, F] to INT8 (swiglu_q8_finish).
template <int NT, int CPG, bool ASYM, bool SPLIT, bool SWIGLU = false, bool GROUPED = false,
          bool SB = false, bool F32 = false, bool Q8 = false, bool F16 = false>
__device__ void w4a16_consumer(const Smem& sm, const GemvArgs& a) {
    static_assert(!(GROUPED && (SPLIT || SWIGLU)), "grouped plans are unsplit, plain epilogue");
    static_assert(!(F32 && (SWIGLU || GROUPED || SB)), "fp32 partial outputs: plain layer only");
    static_assert(!Q8 || (SWIGLU && !GROUPED && !SB && !F32), "INT8 outputs: SwiGLU epilogue only");
    static_assert(!F16 || NT == 1, "the fp16 path takes one token tile");
    constexpr int SEG = 8 / CPG;
    constexpr int LOG_CPG = CPG == 8 ? 3 : CPG == 4 ? 2 : CPG == 2 ? 1 : 0;
    constexpr bool PF = SEG <= 2;           // scales one stage ahead when they are few
    // kernel arguments in registers (asm statements with memory clobbers
    // would otherwise force re-reads from parameter space)
    const int N = a.N, K = a.K, Kp = a.Kp, Ng = a.Ng, SKE = a.SKE, XS = a.XS;
    const int Sp = a.S, spl = a.spl, nst = a.nst, R = a.R;
    int M = GROUPED ? a.gmax : a.M;            // GROUPED: set per group
    int units = a.units;                       // GROUPED: from the list
    const float* __restrict__ scales = a.scales;
    const uint8_t* __restrict__ zeros = a.zeros;
    const float* __restrict__ bias = a.bias;
    uint16_t* __restrict__ y = a.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tig = lane & 3, gid = lane >> 2;
    const int WR = R / 16, WK = CW / WR;
    const int rt = warp % WR, kp = warp / WR;
    const uint16_t* x = static_cast<const uint16_t*>(a.x);
    const uint32_t wbuf_u = smem_u32(sm.wbuf), xbuf_u = smem_u32(sm.xbuf);
    const int lj = lane >> 3, li = lane & 7;
    // this warp's 16 x 256 box inside a stage, and the ldmatrix row and
    // swizzled chunk offset of this lane for each chunk pair
    const uint32_t l_off = (uint32_t)(kp * R * 128 + (rt * 16 + ((lj & 1) << 3) + li) * 128);
    uint32_t l_cp[4];
#pragma unroll
    for (int cp = 0; cp < 4; ++cp) l_cp[cp] = l_off + ((uint32_t)((2 * cp + (lj >> 1)) ^ li) << 4);
    uint32_t xrow[NT];
    int xt[NT][2];                             // F16: this thread's tokens in xseg
    auto token_rows = [&]() {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            xrow[nt] = xbuf_u + (uint32_t)(min(nt * 8 + gid, M - 1) * XS + tig * 16 + kp * 512);
            xt[nt][0] = 4 * min(nt * 8 + 2 * tig, M - 1);
            xt[nt][1] = 4 * min(nt * 8 + 2 * tig + 1, M - 1);
        }
    };
    token_rows();
    // group of a segment: segments of CPG*32 columns tile the groups exactly,
    // so g = segment / (G / (CPG*32)), a shift when that ratio is a power of 2
    const int gdiv = a.G / (CPG * 32);
    // G = 32 with rows of whole 8-group runs: scales and zero points of a
    // box can be read with vector loads (16 B / 8 B aligned)
    const bool vec_groups = gdiv == 1 && (Ng % 8) == 0;
    const int gshift = (gdiv & (gdiv - 1)) == 0 ? __ffs(gdiv) - 1 : -1;
    const float zc[4] = {0.f, 0.f, 0.f, 0.f};
    SmemCtl* ctl = sm.ctl;
    const bool xtma = a.xtma != 0;

    uint32_t it = 0, xi = 0;
    int prev0 = -1, prev1 = -1;
    bool waited = false;
    const int* glist = nullptr;
    int prev_item = -1;
    int inject = 0;                            // GROUPED: failure-test switches
    if constexpr (GROUPED) {
        // (group, token tile) items in group order, the same list in every CTA
        grid_dep_wait();
        waited = true;
        inject = fault_injection_of(a.err);
        int* list = reinterpret_cast<int*>(sm.wbuf + a.list_off);
        int* wcnt = reinterpret_cast<int*>(sm.red);
        int nitems = 0;
        for (int e0 = 0; e0 < a.E; e0 += NCT) {
            const int e = e0 + tid;
            int nt_e = 0;                                    // this group's tiles
            if (e < a.E) {
                const int o0 = __ldg(a.goff + e), o1 = __ldg(a.goff + e + 1);
                const bool valid = o0 >= 0 && o1 >= o0 && o1 <= a.M;
                if (!valid) atomicCAS(a.err, 0, W4_ERR_GROUP_TOKENS);
                nt_e = valid ? (o1 - o0 + a.gmax - 1) / a.gmax : 0;
            }
            int v = nt_e;                                    // inclusive scan in the warp
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            if (lane == 31) wcnt[warp] = v;
            named_bar_sync(1, NCT);
            int before = nitems, tot = 0;
            for (int w = 0; w < CW; ++w) {
                const int c = wcnt[w];
                if (w < warp) before += c;
                tot += c;
            }
            // offsets that overlap can list more tiles than T allows: the
            // list keeps what fits and the error is flagged
            for (int t = 0; t < nt_e; ++t) {
                const int at = before + v - nt_e + t;
                if (at < a.list_cap) list[at] = e | (t << 16);
            }
            nitems += tot;
            named_bar_sync(1, NCT);
        }
        if (nitems > a.list_cap) {
            if (tid == 0) atomicCAS(a.err, 0, W4_ERR_GROUP_TOKENS);
            nitems = a.list_cap;
        }
        if (tid == 0) {
            ctl->nact = nitems;
            if (!(inject & kInjectNoList)) mbar_arrive(&ctl->listready);
        }
        units = nitems * a.NBg;
        glist = list;
    }
    int u_beg = blockIdx.x, u_end = units, u_step = gridDim.x;
    if constexpr (GROUPED) {                   // the producer's contiguous runs
        u_beg = (int)(((long long)units * blockIdx.x) / gridDim.x);
        u_end = (int)(((long long)units * (blockIdx.x + 1)) / gridDim.x);
        u_step = 1;
    }
    for (int u = u_beg; u < u_end; u += u_step) {
        int rb, s, ks0, ks1, g = 0;
        if constexpr (GROUPED) {
            const int gi = u / a.NBg;
            rb = u - gi * a.NBg;
            const int item = glist[gi];
            g = item & 0xFFFF;
            s = 0; ks0 = 0; ks1 = nst;
            if (item != prev_item) {
                // this tile's tokens: rows o0 .. o0 + M - 1 of x and y
                const int o0 = __ldg(a.goff + g) + (item >> 16) * a.gmax;
                M = min(a.gmax, __ldg(a.goff + g + 1) - o0);
                x = static_cast<const uint16_t*>(a.x) + (size_t)o0 * K;
                y = a.y + (size_t)o0 * N;
                token_rows();
                prev0 = -1;                        // stage this tile's activations
                prev_item = item;
            }
        } else {
            rb = u / Sp;
            s = u - rb * Sp;
            ks0 = s * spl;
            ks1 = min(ks0 + spl, nst);
        }
        const size_t wrow = GROUPED ? (size_t)g * N : 0;   // first row of this unit's matrix
        const int row0 = rb * R + rt * 16;
        const int nr = min(row0 + gid, N - 1), nr8 = min(row0 + gid + 8, N - 1);
        // the two rows' parameters: fp32 scales and uint8 zero points, or
        // (SB) bf16 scales and bf16 offsets through the same two pointers
        const float* sc_r = SB ? reinterpret_cast<const float*>(a.scales_b + (wrow + nr) * Ng)
                               : scales + (wrow + nr) * Ng;
        const float* sc_r8 = SB ? reinterpret_cast<const float*>(a.scales_b + (wrow + nr8) * Ng)
                                : scales + (wrow + nr8) * Ng;
        const uint8_t* zp_r = !ASYM ? nullptr
                              : SB ? reinterpret_cast<const uint8_t*>(a.offs_b + (wrow + nr) * Ng)
                                   : zeros + (wrow + nr) * Ng;
        const uint8_t* zp_r8 = !ASYM ? nullptr
                               : SB ? reinterpret_cast<const uint8_t*>(a.offs_b + (wrow + nr8) * Ng)
                                    : zeros + (wrow + nr8) * Ng;
        // bias of this thread's two rows and the scales of the first stage:
        // constant inputs, read before waiting for the previous kernel
        const float b_lo = bias ? __ldg(bias + wrow + nr) : 0.f;
        const float b_hi = bias ? __ldg(bias + wrow + nr8) : 0.f;
        float sr[SEG], sr8[SEG], zr[SEG], zr8[SEG];
        auto load_scales = [&](int kw, float* r_, float* r8_, float* z_, float* z8_) {
            if constexpr (SB) {
                // bf16 scales (z_: offsets); eight 32-wide groups of a box are
                // one 16-byte load per row when aligned and inside the row
                auto bf = [](uint32_t w, int hi) { return __uint_as_float(hi ? (w & 0xFFFF0000u) : (w << 16)); };
                const uint16_t* sb_r = reinterpret_cast<const uint16_t*>(sc_r);
                const uint16_t* sb_r8 = reinterpret_cast<const uint16_t*>(sc_r8);
                const uint16_t* ob_r = reinterpret_cast<const uint16_t*>(zp_r);
                const uint16_t* ob_r8 = reinterpret_cast<const uint16_t*>(zp_r8);
                if constexpr (SEG == 8) {
                    const int g0 = kw >> (5 + LOG_CPG);
                    if (vec_groups && g0 + 8 <= Ng) {
                        const uint4 a4 = __ldg(reinterpret_cast<const uint4*>(sb_r + g0));
                        const uint4 b4 = __ldg(reinterpret_cast<const uint4*>(sb_r8 + g0));
                        const uint32_t aw[4] = {a4.x, a4.y, a4.z, a4.w}, bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            r_[j] = bf(aw[j >> 1], j & 1);
                            r8_[j] = bf(bw[j >> 1], j & 1);
                        }
                        if (ASYM) {
                            const uint4 c4 = __ldg(reinterpret_cast<const uint4*>(ob_r + g0));
                            const uint4 d4 = __ldg(reinterpret_cast<const uint4*>(ob_r8 + g0));
                            const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w}, dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                z_[j] = bf(cw[j >> 1], j & 1);
                                z8_[j] = bf(dw[j >> 1], j & 1);
                            }
                        }
                        return;
                    }
                }
#pragma unroll
                for (int j = 0; j < SEG; ++j) {
                    const int sg = (kw >> (5 + LOG_CPG)) + j;
                    const int g = min(gshift >= 0 ? (sg >> gshift) : sg / gdiv, Ng - 1);
                    r_[j] = __uint_as_float((uint32_t)__ldg(sb_r + g) << 16);
                    r8_[j] = __uint_as_float((uint32_t)__ldg(sb_r8 + g) << 16);
                    if (ASYM) {
                        z_[j] = __uint_as_float((uint32_t)__ldg(ob_r + g) << 16);
                        z8_[j] = __uint_as_float((uint32_t)__ldg(ob_r8 + g) << 16);
                    }
                }
            } else {
                if constexpr (SEG == 8) {
                    // one group per segment (G = 32): a row's 8 scales (32 B) and
                    // zero points (8 B) of the box are contiguous; vector loads
                    // when they are aligned and inside the row
                    const int g0 = kw >> (5 + LOG_CPG);
                    if (vec_groups && g0 + 8 <= Ng) {
                        const float4* s4 = reinterpret_cast<const float4*>(sc_r + g0);
                        const float4* s48 = reinterpret_cast<const float4*>(sc_r8 + g0);
                        const float4 a0 = __ldg(s4), a1 = __ldg(s4 + 1);
                        const float4 b0 = __ldg(s48), b1 = __ldg(s48 + 1);
                        r_[0] = a0.x; r_[1] = a0.y; r_[2] = a0.z; r_[3] = a0.w;
                        r_[4] = a1.x; r_[5] = a1.y; r_[6] = a1.z; r_[7] = a1.w;
                        r8_[0] = b0.x; r8_[1] = b0.y; r8_[2] = b0.z; r8_[3] = b0.w;
                        r8_[4] = b1.x; r8_[5] = b1.y; r8_[6] = b1.z; r8_[7] = b1.w;
                        if (ASYM) {
                            const uint2 q = __ldg(reinterpret_cast<const uint2*>(zp_r + g0));
                            const uint2 q8 = __ldg(reinterpret_cast<const uint2*>(zp_r8 + g0));
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                z_[j] = (float)((q.x >> (8 * j)) & 0xFF);
                                z_[j + 4] = (float)((q.y >> (8 * j)) & 0xFF);
                                z8_[j] = (float)((q8.x >> (8 * j)) & 0xFF);
                                z8_[j + 4] = (float)((q8.y >> (8 * j)) & 0xFF);
                            }
                        }
                        return;
                    }
                }
#pragma unroll
                for (int j = 0; j < SEG; ++j) {
                    const int sg = (kw >> (5 + LOG_CPG)) + j;
                    const int g = min(gshift >= 0 ? (sg >> gshift) : sg / gdiv, Ng - 1);
                    r_[j] = __ldg(sc_r + g);
                    r8_[j] = __ldg(sc_r8 + g);
                    if (ASYM) {
                        z_[j] = (float)__ldg(zp_r + g);
                        z8_[j] = (float)__ldg(zp_r8 + g);
                    }
                }
            }
        };
        if (PF) load_scales(min(ks0 * SKE + kp * 256, Kp - 1), sr, sr8, zr, zr8);
        if (!waited) {
            grid_dep_wait();     // x, the workspace and y come after this point
            waited = true;
        }

        named_bar_sync(1, NCT);
        if (ks0 != prev0 || ks1 != prev1) {
            if (xtma) {
                // everyone is past the previous slice: release its buffer,
                // then wait for this slice's copy and zero its tail
                if (xi > 0 && tid == 0) {
                    fence_proxy_async_smem();     // zero tails written here, then the copy
                    mbar_arrive(&ctl->xempty);
                }
                if (mbar_wait(&ctl->xfull, xi & 1, &ctl->abort, a.err)) {
                    if constexpr (F16)
                        stage_x_f16<CPG, true, SPLIT ? 2 : 4>(sm.xbuf, sm.xseg, x, M, K, XS,
                                                             ks0 * SKE, (ks1 - ks0) * SKE, tid);
                    else
                        stage_x_bf16<true>(sm.xbuf, x, M, K, XS, ks0 * SKE, (ks1 - ks0) * SKE, tid);
                }
                ++xi;
            } else if constexpr (F16) {
                stage_x_f16<CPG, false, SPLIT ? 2 : 4>(sm.xbuf, sm.xseg, x, M, K, XS, ks0 * SKE,
                                                      (ks1 - ks0) * SKE, tid);
            } else {
                stage_x_bf16<false>(sm.xbuf, x, M, K, XS, ks0 * SKE, (ks1 - ks0) * SKE, tid);
            }
            named_bar_sync(1, NCT);
            prev0 = ks0;
            prev1 = ks1;
        }

        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[nt][j] = 0.f;

        // bf16 path: the MMA sums (c - z) x over each run of CPG chunks (one
        // group), c - z exact in bf16 (the 128 + z offsets are subtracted from
        // the unpacked words), x the bf16 activations as they are: tmp = sum
        // (c - z) x, every product exact in fp32, and acc += s * tmp.  SB with
        // offsets: c - 8 in place of c - z, and a second MMA with weights 1
        // gives C1 = sum x, so acc += s * tmp + o * C1.
        // F16 path: the MMA sums x' * w' with w' = 1024 + c on even and
        // 1024 + 16c on odd columns and x' the segment's scaled activations
        // (odd ones / 16); with the segment's (u, C0, C1) from staging,
        // acc += s * (u * tmp - C0 - z * C1).

        for (int ks = ks0; ks < ks1; ++ks, ++it) {
            const int slot = it % NS;
            const int kw = ks * SKE + kp * 256;            // first column of this warp's box
            float nsr[SEG], nsr8[SEG], nzr[SEG], nzr8[SEG];
            if (PF && ks + 1 < ks1)
                load_scales(min(kw + SKE, Kp - 1), nsr, nsr8, nzr, nzr8);
            if (kw < Kp) {
                if (!PF) load_scales(kw, sr, sr8, zr, zr8);
                if (mbar_wait(&ctl->full[slot], (it / NS) & 1, &ctl->abort, a.err)) {
                    const uint32_t wst = wbuf_u + slot * STAGE_BYTES;
                    const uint32_t xoff = (uint32_t)(ks - ks0) * (uint32_t)(SKE * 2);
                    if constexpr (F16) {
                        const float* xs_st =
                            sm.xseg + 4 * ((((ks - ks0) * SKE + kp * 256) >> (5 + LOG_CPG)) * M);
                        float tmp[NT][4];
#pragma unroll
                        for (int cp = 0; cp < 4; ++cp) {
                            uint32_t r[4];
                            ldmatrix_x4_nc(wst + l_cp[cp], r[0], r[1], r[2], r[3]);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int c = 2 * cp + h;
                                const int seg = c / CPG;
                                uint32_t P[4], Q[4];
                                nibbles_to_f16x2_biased(r[2 * h], P);
                                nibbles_to_f16x2_biased(r[2 * h + 1], Q);
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    uint32_t X[4];
                                    lds128(xrow[nt] + xoff + c * 64, X);
                                    mma_f16_16816(tmp[nt], P[0], Q[0], P[1], Q[1], X[0], X[1],
                                                  (c % CPG == 0) ? zc : tmp[nt]);
                                    mma_f16_16816(tmp[nt], P[2], Q[2], P[3], Q[3], X[2], X[3], tmp[nt]);
                                }
                                if ((c + 1) % CPG == 0) {
#pragma unroll
                                    for (int nt = 0; nt < NT; ++nt) {
                                        const float4 e0 = *reinterpret_cast<const float4*>(
                                            xs_st + 4 * seg * M + xt[nt][0]);
                                        const float4 e1 = *reinterpret_cast<const float4*>(
                                            xs_st + 4 * seg * M + xt[nt][1]);
                                        float c00, c01, c10, c11;   // C0 + z C1 per (row, token)
                                        if (ASYM && !SB) {
                                            c00 = fmaf(zr[seg], e0.z, e0.y);
                                            c01 = fmaf(zr[seg], e1.z, e1.y);
                                            c10 = fmaf(zr8[seg], e0.z, e0.y);
                                            c11 = fmaf(zr8[seg], e1.z, e1.y);
                                        } else {
                                            c00 = c10 = fmaf(8.f, e0.z, e0.y);
                                            c01 = c11 = fmaf(8.f, e1.z, e1.y);
                                        }
                                        if (ASYM && SB) {           // + o C1 (zr: offsets)
                                            acc[nt][0] = fmaf(zr[seg], e0.z, acc[nt][0]);
                                            acc[nt][1] = fmaf(zr[seg], e1.z, acc[nt][1]);
                                            acc[nt][2] = fmaf(zr8[seg], e0.z, acc[nt][2]);
                                            acc[nt][3] = fmaf(zr8[seg], e1.z, acc[nt][3]);
                                        }
                                        acc[nt][0] = fmaf(sr[seg], fmaf(e0.x, tmp[nt][0], -c00), acc[nt][0]);
                                        acc[nt][1] = fmaf(sr[seg], fmaf(e1.x, tmp[nt][1], -c01), acc[nt][1]);
                                        acc[nt][2] = fmaf(sr8[seg], fmaf(e0.x, tmp[nt][2], -c10), acc[nt][2]);
                                        acc[nt][3] = fmaf(sr8[seg], fmaf(e1.x, tmp[nt][3], -c11), acc[nt][3]);
                                    }
                                }
                            }
                        }
                    } else {
                        float tmp[NT][4];
                        float c1[(ASYM && SB) ? NT : 1][4];
#pragma unroll
                        for (int cp = 0; cp < 4; ++cp) {
                            uint32_t r[4];
                            ldmatrix_x4_nc(wst + l_cp[cp], r[0], r[1], r[2], r[3]);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int c = 2 * cp + h;
                                const int seg = c / CPG;
                                // bf16 pairs 128 + z of the two rows (z = 8 unless ASYM && !SB)
                                uint32_t o = 0x43084308u, oh = 0x43084308u;
                                if constexpr (ASYM && !SB) {
                                    o = (0x4300u + (uint32_t)(int)zr[seg]) * 0x10001u;
                                    oh = (0x4300u + (uint32_t)(int)zr8[seg]) * 0x10001u;
                                }
                                // thread tig holds codes k = 8 tig .. 8 tig + 7 of the
                                // chunk (rows gid, gid + 8) and reads x at the same k
                                uint32_t P[4], Q[4];
                                nibbles_to_bf16x2_pairs(r[2 * h], P);
                                nibbles_to_bf16x2_pairs(r[2 * h + 1], Q);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    P[i] = sub_bf16x2(P[i], o);
                                    Q[i] = sub_bf16x2(Q[i], oh);
                                }
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    uint32_t X[4];
                                    lds128(xrow[nt] + xoff + c * 64, X);
                                    mma_bf16_16816(tmp[nt], P[0], Q[0], P[1], Q[1], X[0], X[1],
                                                   (c % CPG == 0) ? zc : tmp[nt]);
                                    mma_bf16_16816(tmp[nt], P[2], Q[2], P[3], Q[3], X[2], X[3], tmp[nt]);
                                    if constexpr (ASYM && SB) {
                                        const uint32_t one = 0x3F803F80u;          // bf16 pairs (1, 1)
                                        mma_bf16_16816(c1[nt], one, one, one, one, X[0], X[1],
                                                       (c % CPG == 0) ? zc : c1[nt]);
                                        mma_bf16_16816(c1[nt], one, one, one, one, X[2], X[3], c1[nt]);
                                    }
                                }
                                if ((c + 1) % CPG == 0) {
#pragma unroll
                                    for (int nt = 0; nt < NT; ++nt) {
                                        if constexpr (ASYM && SB) {       // + o C1 (zr: offsets)
                                            acc[nt][0] = fmaf(zr[seg], c1[nt][0], acc[nt][0]);
                                            acc[nt][1] = fmaf(zr[seg], c1[nt][1], acc[nt][1]);
                                            acc[nt][2] = fmaf(zr8[seg], c1[nt][2], acc[nt][2]);
                                            acc[nt][3] = fmaf(zr8[seg], c1[nt][3], acc[nt][3]);
                                        }
                                        acc[nt][0] = fmaf(sr[seg], tmp[nt][0], acc[nt][0]);
                                        acc[nt][1] = fmaf(sr[seg], tmp[nt][1], acc[nt][1]);
                                        acc[nt][2] = fmaf(sr8[seg], tmp[nt][2], acc[nt][2]);
                                        acc[nt][3] = fmaf(sr8[seg], tmp[nt][3], acc[nt][3]);
                                    }
                                }
                            }
                        }
                    }
                }
            }
            if (PF) {
#pragma unroll
                for (int j = 0; j < SEG; ++j) {
                    sr[j] = nsr[j]; sr8[j] = nsr8[j];
                    if (ASYM) { zr[j] = nzr[j]; zr8[j] = nzr8[j]; }
                }
            }
            __syncwarp();
            if (lane == 0 && !(GROUPED && (inject & kInjectNoRelease))) mbar_arrive(&ctl->empty[slot]);
        }

        // ---- add the k-phases of each row tile, in order 0, 1, ..., WK-1
        if (WK > 1) {
            if (kp > 0) {
                float* dst = sm.red + ((kp - 1) * WR + rt) * (NT * 4 * 32) + lane;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 4; ++j) dst[(nt * 4 + j) * 32] = acc[nt][j];
            }
            named_bar_sync(1, NCT);
            if (kp == 0) {
                for (int q = 1; q < WK; ++q) {
                    const float* src = sm.red + ((q - 1) * WR + rt) * (NT * 4 * 32) + lane;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[nt][j] += src[(nt * 4 + j) * 32];
                }
            }
        }

        // ---- cluster split: ranks 1..S-1 store their sums into rank 0's
        // receive buffer (slot s-1, the register layout of the k-phase
        // buffer) and arrive on its barrier; rank 0 adds them in split order
        // and writes y like an unsplit plan.  One unit per CTA.
        bool direct = !SPLIT;                  // this CTA writes y from acc
        // (not compiled into the fp16-loop instances, whose 1-2 token plans
        // never take it: left out, their code stays as measured)
        if constexpr (SPLIT && !F16) {
            if (a.csplit) {
                const int slot_floats = WR * NT * 4 * 32;
                float* recv = reinterpret_cast<float*>(sm.wbuf + a.crecv_off);
                const int idx0 = rt * (NT * 4 * 32) + lane;
                if (s > 0) {
                    if (kp == 0) {
                        const uint32_t dst = mapa_shared(smem_u32(recv + (s - 1) * slot_floats + idx0), 0);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                st_shared_cluster(dst + 4u * (uint32_t)((nt * 4 + j) * 32), acc[nt][j]);
                    }
                    named_bar_sync(1, NCT);
                    if (tid == 0) mbar_arrive_release_cluster(mapa_shared(smem_u32(&ctl->cready), 0));
                } else {
                    direct = mbar_wait_cluster(&ctl->cready, 0, &ctl->abort, a.err);
                    // after an abort elsewhere, still let the other ranks'
                    // stores into this CTA land before it can exit
                    if (!direct) mbar_wait_drain(&ctl->cready, 0, a.err);
                    if (direct && kp == 0) {
                        for (int q = 1; q < Sp; ++q) {
                            const float* src = recv + (q - 1) * slot_floats + idx0;
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int j = 0; j < 4; ++j) acc[nt][j] += src[(nt * 4 + j) * 32];
                        }
                    }
                }
            }
        }

        // ---- epilogue: thread holds (token 8nt + 2tig + (j&1), row gid + 8(j>>1))
        if (direct) {
        if constexpr (SWIGLU) {
            if (kp == 0) {
                const int F = N >> 1, f = (row0 >> 1) + gid;       // this lane's output column
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int t = nt * 8 + 2 * tig + j;
                        const float v = swiglu(acc[nt][j] + b_lo, acc[nt][j + 2] + b_hi);
                        if (t < M && row0 + gid < N) y[(size_t)t * F + f] = f32_to_bf16_bits(v);
                        if constexpr (Q8) q8_cta_max(ctl, v, t, M, lane, t < M && row0 + gid < N);
                    }
            }
        } else {
            if (kp == 0) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int t = nt * 8 + 2 * tig + (j & 1);
                        const int n = row0 + gid + 8 * (j >> 1);
                        if (t < M && n < N) {
                            if constexpr (F32) a.y32[(size_t)t * N + n] = acc[nt][j];
                            else y[(size_t)t * N + n] = f32_to_bf16_bits(acc[nt][j] + ((j >> 1) ? b_hi : b_lo));
                        }
                    }
            }
        }
        } else if (SPLIT && (F16 || !a.csplit)) {
            float* part = static_cast<float*>(a.partial);
            if (kp == 0) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int t = nt * 8 + 2 * tig + (j & 1);
                        const int n = row0 + gid + 8 * (j >> 1);
                        if (t < M && n < N) part[((size_t)s * M + t) * N + n] = acc[nt][j];
                    }
            }
            if (split_k_arrive(a, ctl, rb)) {
                if (kp == 0) {
                    if constexpr (SWIGLU) {
                        const int F = N >> 1, f = (row0 >> 1) + gid;
                        const int ng = row0 + gid, nu = ng + 8;   // gate and up rows
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const int t = nt * 8 + 2 * tig + j;
                                float v = 0.f;
                                if (t < M && ng < N) {
                                    const float g = sum_splits(part + (size_t)t * N + ng, (size_t)M * N, Sp);
                                    const float u = sum_splits(part + (size_t)t * N + nu, (size_t)M * N, Sp);
                                    v = swiglu(g + b_lo, u + b_hi);
                                    y[(size_t)t * F + f] = f32_to_bf16_bits(v);
                                }
                                if constexpr (Q8) q8_cta_max(ctl, v, t, M, lane, t < M && ng < N);
                            }
                    } else {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int t = nt * 8 + 2 * tig + (j & 1);
                            const int n = row0 + gid + 8 * (j >> 1);
                            if (t < M && n < N) {
                                const float v = sum_splits(part + (size_t)t * N + n, (size_t)M * N, Sp);
                                if constexpr (F32) a.y32[(size_t)t * N + n] = v;
                                else y[(size_t)t * N + n] = f32_to_bf16_bits(v + ((j >> 1) ? b_hi : b_lo));
                            }
                        }
                    }
                }
                if (tid == 0) a.tickets[rb] = 0;
            }
        }
    }
    // (eight loads in flight fit the registers of the one-tile kernels)
    if constexpr (Q8) swiglu_q8_finish<NT == 1 ? 8 : 4>(a, ctl, sm.red, tid);
}

template <int MT>
__device__ void w4a8_consumer(const Smem& sm, const GemvArgs& a) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tig = lane & 3, gid = lane >> 2;
    const int WR = a.R / 16, WK = CW / WR;
    const int rt = warp % WR, kp = warp / WR;
    const int8_t* qx = static_cast<const int8_t*>(a.x);
    const uint32_t wbuf_u = smem_u32(sm.wbuf), xbuf_u = smem_u32(sm.xbuf);
    const int lj = lane >> 3, li = lane & 7;
    const uint32_t l_off = (uint32_t)(kp * a.R * 128 + (rt * 16 + ((lj & 1) << 3) + li) * 128);
    uint32_t l_cp[4];
#pragma unroll
    for (int cp = 0; cp < 4; ++cp) l_cp[cp] = l_off + ((uint32_t)((2 * cp + (lj >> 1)) ^ li) << 4);
    uint32_t xrow[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m)
        xrow[m] = xbuf_u + (uint32_t)(min(m, a.M - 1) * a.XS + tig * 8 + kp * 256);
    int* red = reinterpret_cast<int*>(sm.red);

    grid_dep_wait();
    uint32_t it = 0;
    int prev0 = -1, prev1 = -1;
    for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
        int rb, s, ks0, ks1;
        unit_coords(u, a, rb, s, ks0, ks1);
        const int row0 = rb * a.R + rt * 16;

        named_bar_sync(1, NCT);
        if (ks0 != prev0 || ks1 != prev1) {
            if (tid < 16) sm.ctl->sumq[tid] = 0;
            named_bar_sync(1, NCT);
            stage_x_s8(sm.xbuf, sm.ctl, qx, a.M, a.Kp, a.XS, ks0 * a.SKE, (ks1 - ks0) * a.SKE, tid);
            named_bar_sync(1, NCT);
            prev0 = ks0;
            prev1 = ks1;
        }

        int acc[MT][2];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = 0;

        for (int ks = ks0; ks < ks1; ++ks, ++it) {
            const int slot = it % NS;
            const int kw = ks * a.SKE + kp * 256;
            if (kw < a.Kp &&
                mbar_wait(&sm.ctl->full[slot], (it / NS) & 1, &sm.ctl->abort, a.err)) {
                const uint32_t wst = wbuf_u + slot * STAGE_BYTES;
                const uint32_t xoff = (uint32_t)(ks - ks0) * (uint32_t)a.SKE;
#pragma unroll
                for (int cp = 0; cp < 4; ++cp) {
                    uint32_t r[4];
                    ldmatrix_x4(wst + l_cp[cp], r[0], r[1], r[2], r[3]);
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
            if (lane == 0) mbar_arrive(&sm.ctl->empty[slot]);
        }

        // lanes sharing a row, then the k-phases (exact integers)
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                int v = acc[m][h];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                acc[m][h] = v;
            }
        if (WK > 1) {
            if (kp > 0) {
                int* dst = red + ((kp - 1) * WR + rt) * (MT * 2 * 32) + lane;
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int h = 0; h < 2; ++h) dst[(m * 2 + h) * 32] = acc[m][h];
            }
            named_bar_sync(1, NCT);
            if (kp == 0) {
                for (int q = 1; q < WK; ++q) {
                    const int* src = red + ((q - 1) * WR + rt) * (MT * 2 * 32) + lane;
#pragma unroll
                    for (int m = 0; m < MT; ++m)
#pragma unroll
                        for (int h = 0; h < 2; ++h) acc[m][h] += src[(m * 2 + h) * 32];
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h) acc[m][h] -= 8 * sm.ctl->sumq[min(m, a.M - 1)];

        int32_t* part = static_cast<int32_t*>(a.partial);
        bool write = kp == 0;
        if (a.S > 1) {
            if (kp == 0) {
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int n = row0 + gid + 8 * h;
                        if (m < a.M && (m & 3) == tig && n < a.N)
                            part[((size_t)s * a.M + m) * a.N + n] = acc[m][h];
                    }
            }
            const bool last = split_k_arrive(a, sm.ctl, rb);
            write = write && last;
            if (last && tid == 0) a.tickets[rb] = 0;
        }
        if (write) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int n = row0 + gid + 8 * h;
                    if (m < a.M && (m & 3) == tig && n < a.N) {
                        int v = acc[m][h];
                        if (a.S > 1) v = sum_splits(part + (size_t)m * a.N + n, (size_t)a.M * a.N, a.S);
                        if (a.acc_out) a.acc_out[(size_t)m * a.N + n] = v;
                        const float sc = __ldg(a.scales + n) * __ldg(a.sx + m);
                        const float b = a.bias ? __ldg(a.bias + n) : 0.f;
                        a.y[(size_t)m * a.N + n] = f32_to_bf16_bits(fmaf(sc, (float)v, b));
                    }
                }
        }
    }
}

// Group-wise W4A8 ("【infra之路】12-投机解码、量化与推理引擎对比", section 2.2
// rule per group; the per-row layout of w4a8_consumer otherwise): for each
// group g of G columns the integer acc_g = sum (code - 8) q_x is formed from
// dp4a partials, y = s_x * sum_g s_W[n, g] acc_g + b.  CPGW = min(G / 32, 8)
// chunks of 32 columns per group inside a warp's 256-column box (G = 32, 64,
// 128, or a multiple of 256: one group per box).  Each lane keeps, per
// (token, row), the integer sums of its 8 columns of the current group,
// sum code * q and sum q, and at the group's last chunk folds
// s_g * (sum code * q - 8 sum q) into an fp32 accumulator; the lanes of a row
// and the k-phase warps then add floats, and K splits add float partials.
// The box's group scales are loaded before its stage's barrier wait.
template <int MT, int CPGW>
__device__ void w4a8g_consumer(const Smem& sm, const GemvArgs& a) {
    constexpr int GPB = 8 / CPGW;                 // groups per 256-column box
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tig = lane & 3, gid = lane >> 2;
    const int WR = a.R / 16, WK = CW / WR;
    const int rt = warp % WR, kp = warp / WR;
    const int Ng = a.Ng;
    const int8_t* qx = static_cast<const int8_t*>(a.x);
    const uint32_t wbuf_u = smem_u32(sm.wbuf), xbuf_u = smem_u32(sm.xbuf);
    const int lj = lane >> 3, li = lane & 7;
    const uint32_t l_off = (uint32_t)(kp * a.R * 128 + (rt * 16 + ((lj & 1) << 3) + li) * 128);
    uint32_t l_cp[4];
#pragma unroll
    for (int cp = 0; cp < 4; ++cp) l_cp[cp] = l_off + ((uint32_t)((2 * cp + (lj >> 1)) ^ li) << 4);
    uint32_t xrow[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m)
        xrow[m] = xbuf_u + (uint32_t)(min(m, a.M - 1) * a.XS + tig * 8 + kp * 256);
    float* red = sm.red;

    grid_dep_wait();
    uint32_t it = 0;
    int prev0 = -1, prev1 = -1;
    for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
        int rb, s, ks0, ks1;
        unit_coords(u, a, rb, s, ks0, ks1);
        const int row0 = rb * a.R + rt * 16;
        const float* sc_lo = a.scales + (size_t)min(row0 + gid, a.N - 1) * Ng;
        const float* sc_hi = a.scales + (size_t)min(row0 + gid + 8, a.N - 1) * Ng;

        named_bar_sync(1, NCT);
        if (ks0 != prev0 || ks1 != prev1) {
            if (tid < 16) sm.ctl->sumq[tid] = 0;
            named_bar_sync(1, NCT);
            stage_x_s8(sm.xbuf, sm.ctl, qx, a.M, a.Kp, a.XS, ks0 * a.SKE, (ks1 - ks0) * a.SKE, tid);
            named_bar_sync(1, NCT);
            prev0 = ks0;
            prev1 = ks1;
        }

        float accf[MT][2];
#pragma unroll
        for (int m = 0; m < MT; ++m) accf[m][0] = accf[m][1] = 0.f;

        for (int ks = ks0; ks < ks1; ++ks, ++it) {
            const int slot = it % NS;
            const int kw = ks * a.SKE + kp * 256;
            if (kw < a.Kp) {
                // this box's groups g0 .. g0 + GPB - 1 (past Ng: zero-filled columns)
                const int g0 = kw / a.G;
                float s_lo[GPB], s_hi[GPB];
#pragma unroll
                for (int j = 0; j < GPB; ++j) {
                    s_lo[j] = g0 + j < Ng ? __ldg(sc_lo + g0 + j) : 0.f;
                    s_hi[j] = g0 + j < Ng ? __ldg(sc_hi + g0 + j) : 0.f;
                }
                if (mbar_wait(&sm.ctl->full[slot], (it / NS) & 1, &sm.ctl->abort, a.err)) {
                    const uint32_t wst = wbuf_u + slot * STAGE_BYTES;
                    const uint32_t xoff = (uint32_t)(ks - ks0) * (uint32_t)a.SKE;
                    int accg[MT][2], sq[MT];
#pragma unroll
                    for (int m = 0; m < MT; ++m) accg[m][0] = accg[m][1] = sq[m] = 0;
#pragma unroll
                    for (int cp = 0; cp < 4; ++cp) {
                        uint32_t r[4];
                        ldmatrix_x4(wst + l_cp[cp], r[0], r[1], r[2], r[3]);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int c = 2 * cp + h;
                            const uint32_t lo = r[2 * h] & 0x0F0F0F0Fu, hi = (r[2 * h] >> 4) & 0x0F0F0F0Fu;
                            const uint32_t lo8 = r[2 * h + 1] & 0x0F0F0F0Fu, hi8 = (r[2 * h + 1] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                uint32_t xe, xo;
                                lds64(xrow[m] + xoff + c * 32, xe, xo);
                                accg[m][0] = dp4a_us(lo, xe, accg[m][0]);
                                accg[m][0] = dp4a_us(hi, xo, accg[m][0]);
                                accg[m][1] = dp4a_us(lo8, xe, accg[m][1]);
                                accg[m][1] = dp4a_us(hi8, xo, accg[m][1]);
                                sq[m] = __dp4a((int)xe, 0x01010101, sq[m]);
                                sq[m] = __dp4a((int)xo, 0x01010101, sq[m]);
                            }
                            if ((c + 1) % CPGW == 0) {         // last chunk of group c / CPGW
                                const int j = c / CPGW;
#pragma unroll
                                for (int m = 0; m < MT; ++m) {
                                    accf[m][0] = fmaf(s_lo[j], (float)(accg[m][0] - 8 * sq[m]), accf[m][0]);
                                    accf[m][1] = fmaf(s_hi[j], (float)(accg[m][1] - 8 * sq[m]), accf[m][1]);
                                    accg[m][0] = accg[m][1] = sq[m] = 0;
                                }
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.ctl->empty[slot]);
        }

        // lanes sharing a row, then the k-phases (fp32 partials)
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v = accf[m][h];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                accf[m][h] = v;
            }
        if (WK > 1) {
            if (kp > 0) {
                float* dst = red + ((kp - 1) * WR + rt) * (MT * 2 * 32) + lane;
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int h = 0; h < 2; ++h) dst[(m * 2 + h) * 32] = accf[m][h];
            }
            named_bar_sync(1, NCT);
            if (kp == 0) {
                for (int q = 1; q < WK; ++q) {
                    const float* src = red + ((q - 1) * WR + rt) * (MT * 2 * 32) + lane;
#pragma unroll
                    for (int m = 0; m < MT; ++m)
#pragma unroll
                        for (int h = 0; h < 2; ++h) accf[m][h] += src[(m * 2 + h) * 32];
                }
            }
        }

        float* part = static_cast<float*>(a.partial);
        bool write = kp == 0;
        if (a.S > 1) {
            if (kp == 0) {
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int n = row0 + gid + 8 * h;
                        if (m < a.M && (m & 3) == tig && n < a.N)
                            part[((size_t)s * a.M + m) * a.N + n] = accf[m][h];
                    }
            }
            const bool last = split_k_arrive(a, sm.ctl, rb);
            write = write && last;
            if (last && tid == 0) a.tickets[rb] = 0;
        }
        if (write) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int n = row0 + gid + 8 * h;
                    if (m < a.M && (m & 3) == tig && n < a.N) {
                        float v = accf[m][h];
                        if (a.S > 1) v = sum_splits(part + (size_t)m * a.N + n, (size_t)a.M * a.N, a.S);
                        const float b = a.bias ? __ldg(a.bias + n) : 0.f;
                        a.y[(size_t)m * a.N + n] = f32_to_bf16_bits(fmaf(__ldg(a.sx + m), v, b));
                    }
                }
        }
    }
}

template <int MT, int CPGW>
__device__ __forceinline__ void w4a8g_body(const CUtensorMap* tm, const GemvArgs& a) {
    const Smem sm = gemv_init(tm, a);
    if (threadIdx.x >= NCT) {
        if (threadIdx.x == NCT) gemv_producer(tm, sm.wbuf, sm.xbuf, sm.ctl, a);
    } else {
        w4a8g_consumer<MT, CPGW>(sm, a);
    }
}

template <int MT, int CPGW>
__global__ void __launch_bounds__(kGemvThreads, 2)
k_w4a8g_gemv_m4(const __grid_constant__ CUtensorMap tmW, const GemvArgs a) {
    w4a8g_body<MT, CPGW>(&tmW, a);
}

template <int MT, int CPGW>
__global__ void __launch_bounds__(kGemvThreads, 1)
k_w4a8g_gemv_m16(const __grid_constant__ CUtensorMap tmW, const GemvArgs a) {
    w4a8g_body<MT, CPGW>(&tmW, a);
}

// Kernel instances that the plan may place two to an SM (M <= 8 for W4A16,
// M <= 4 for W4A8) are compiled for two resident CTAs of 288 threads.
template <int NT, int CPG, bool ASYM, bool SPLIT, bool SWIGLU, bool GROUPED, bool SB, bool F32,
          bool Q8, bool F16 = false>
__device__ __forceinline__ void w4a16_body(const CUtensorMap* tm, const GemvArgs& a) {
    const Smem sm = gemv_init<GROUPED>(tm, a);
    if (threadIdx.x >= NCT) {
        if (threadIdx.x == NCT) gemv_producer<GROUPED>(tm, sm.wbuf, sm.xbuf, sm.ctl, a);
    } else {
        w4a16_consumer<NT, CPG, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8, F16>(sm, a);
    }
}

// One token tile on the fp16 path (1 or 2 tokens, groups of 64 or more).
template <int CPG, bool ASYM, bool SPLIT, bool SWIGLU, bool GROUPED = false, bool SB = false,
          bool F32 = false, bool Q8 = false>
__global__ void __launch_bounds__(kGemvThreads, 2)
k_w4a16_gemv_m2(const __grid_constant__ CUtensorMap tmW, const GemvArgs a) {
    w4a16_body<1, CPG, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8, true>(&tmW, a);
}

template <int CPG, bool ASYM, bool SPLIT, bool SWIGLU, bool GROUPED = false, bool SB = false,
          bool F32 = false, bool Q8 = false>
__global__ void __launch_bounds__(kGemvThreads, 2)
k_w4a16_gemv_m8(const __grid_constant__ CUtensorMap tmW, const GemvArgs a) {
    w4a16_body<1, CPG, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>(&tmW, a);
}

template <int CPG, bool ASYM, bool SPLIT, bool SWIGLU, bool GROUPED = false, bool SB = false,
          bool F32 = false, bool Q8 = false>
__global__ void __launch_bounds__(kGemvThreads, 1)
k_w4a16_gemv_m16(const __grid_constant__ CUtensorMap tmW, const GemvArgs a) {
    w4a16_body<2, CPG, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>(&tmW, a);
}

template <int MT>
__device__ __forceinline__ void w4a8_body(const CUtensorMap* tm, const GemvArgs& a) {
    const Smem sm = gemv_init(tm, a);
    if (threadIdx.x >= NCT) {
        if (threadIdx.x == NCT) gemv_producer(tm, sm.wbuf, sm.xbuf, sm.ctl, a);
    } else {
        w4a8_consumer<MT>(sm, a);
    }
}

template <int MT>
__global__ void __launch_bounds__(kGemvThreads, 2)
k_w4a8_gemv_m4(const __grid_constant__ CUtensorMap tmW, const GemvArgs a) {
    w4a8_body<MT>(&tmW, a);
}

template <int MT>
__global__ void __launch_bounds__(kGemvThreads, 1)
k_w4a8_gemv_m16(const __grid_constant__ CUtensorMap tmW, const GemvArgs a) {
    w4a8_body<MT>(&tmW, a);
}

// Largest dynamic shared memory set so far per (kernel, device).
inline bool raise_smem_limit(const void* kern, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, size_t> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lk(mu);
    size_t& cur = done[{kern, dev}];
    if (bytes <= cur) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
        cudaSuccess)
        return false;
    cur = bytes;
    return true;
}

// Whether `grid` CTAs in clusters of S fit on the device at once with this
// launch's shared memory (cached per kernel, device, size and S).
template <typename Kern>
bool clusters_fit(const void* key, Kern kern, const cudaLaunchConfig_t& cfg, int S, int grid) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, size_t, int>, int> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lk(mu);
    const auto k = std::make_tuple(key, dev, cfg.dynamicSmemBytes, S);
    auto it = done.find(k);
    if (it == done.end()) {
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        it = done.emplace(k, n).first;
    }
    return (long long)it->second * S >= grid;
}

template <typename Kern>
int launch(Kern kern, const uint8_t* packed, const GemvArgs& a0, const GemvPlan& p,
           cudaStream_t stream) {
    GemvArgs a = a0;
    // stages of the first unit prefetched into L2 before the dependency wait
    // (W4_GEMV_PF, 0..4).  W4A16: one, measured on the 7B step at one token:
    // the prefetches compete with the previous kernel's tail and this
    // kernel's activation reads, so a deeper prefetch that helps a linear
    // alone (two stages: gate_up 14.8 -> 14.4 us) slows the chain (0: 3,516
    // GB/s, 1: 3,698, 2: 3,659, 3: 3,581, 4: 3,533).  W4A8 (a.sx set): the
    // whole ring, since its predecessor is the short activation quantizer
    // (with one stage the quantizer + up pair went from 8.3 to 9.3 us)
    {
        const char* e = std::getenv("W4_GEMV_PF");
        a.pf = e ? std::max(0, std::min(NS, std::atoi(e))) : (a0.sx ? NS : 1);
        // the hold (W4_GEMV_XFIRST=n stages before it, -1 none) exists only
        // on the fp16 path with the activations read by the consumers, whose
        // staging writes the per-segment sums it watches.  Default 2 (the
        // last stage of the 3-deep ring waits), measured on the 7B step at
        // one token: no hold 3,723 / 3,710 GB/s, after 1 stage 3,660 /
        // 3,656, after 2 3,764 / 3,758 (gate_up 14.7 -> 14.35 us, down 11.76
        // -> 11.28; qkv and o, two stages a CTA, are not held)
        const char* ex = std::getenv("W4_GEMV_XFIRST");
        a.xfirst = (!a0.sx && a0.E <= 0 && p.f16 && !a0.xtma)
                       ? (ex ? std::max(-1, std::atoi(ex)) : 2)
                       : -1;
    }
    CUtensorMap tm;
    // grouped launches stack the E groups' rows
    const uint64_t rows = (uint64_t)a.N * (uint64_t)(a.E > 0 ? a.E : 1);
    if (!encode_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, packed, (uint64_t)(a.Kp / 2),
                        rows, (uint64_t)(a.Kp / 2), 128, (uint32_t)p.R,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return W4_ERR_CUDA;
    // the dynamic shared-memory limit of this kernel, raised only when a plan
    // needs more than was set before for this kernel on this device (one
    // driver call per kernel and size, not per launch)
    if (!raise_smem_limit(reinterpret_cast<const void*>(kern), p.smem)) return W4_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    a.csplit = 0;
    if (a0.coop) {
        // the INT8 epilogue's grid-wide hand-off needs every CTA resident:
        // a cooperative launch (with programmatic launch where the driver
        // accepts both; the outcome is remembered per kernel and device),
        // else a plain launch whose last CTA quantizes alone
        static std::mutex mu;
        static std::map<std::pair<const void*, int>, int> mode;   // 1 coop+PDL, 2 coop, 3 plain
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return W4_ERR_CUDA;
        int m;
        {
            std::lock_guard<std::mutex> lk(mu);
            m = mode[{reinterpret_cast<const void*>(kern), dev}];
        }
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
        for (int mt = m ? m : 1; mt <= 3; ++mt) {
            a.coop = mt < 3 ? 1 : 0;
            if (mt == 1) {
                cfg.attrs = attr;
                cfg.numAttrs = 2;
            } else if (mt == 2) {
                cfg.attrs = attr + 1;
                cfg.numAttrs = 1;
            } else {
                cfg.attrs = attr;
                cfg.numAttrs = 1;
            }
            if (cudaLaunchKernelEx(&cfg, kern, tm, a) == cudaSuccess) {
                std::lock_guard<std::mutex> lk(mu);
                mode[{reinterpret_cast<const void*>(kern), dev}] = mt;
                return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
            }
            cudaGetLastError();
        }
        return W4_ERR_CUDA;
    }
    if (p.csplit) {
        // clusters of the S splits of a row block, when the whole grid fits
        // on the GPU at once as clusters (else the global hand-off, which the
        // same kernel and workspace also support)
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)p.S;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        if (clusters_fit(reinterpret_cast<const void*>(kern), kern, cfg, p.S, p.grid)) {
            a.csplit = 1;
            a.crecv_off = (int)p.crecv_off;
        } else {
            cfg.numAttrs = 1;
        }
    }
    if (cudaLaunchKernelEx(&cfg, kern, tm, a) != cudaSuccess) return W4_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

template <int NT, bool ASYM, bool SPLIT, bool SWIGLU = false, bool GROUPED = false,
          bool SB = false, bool F32 = false, bool Q8 = false>
int launch_w4a16_cpg(int cpg, const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                     cudaStream_t st) {
    if (NT == 1 && p.f16) {
        switch (cpg) {
            case 8: return launch(k_w4a16_gemv_m2<8, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>, packed, a, p, st);
            case 4: return launch(k_w4a16_gemv_m2<4, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>, packed, a, p, st);
            case 2: return launch(k_w4a16_gemv_m2<2, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>, packed, a, p, st);
            default: return W4_ERR_UNSUPPORTED_GROUP;
        }
    }
    if (NT == 1) {
        switch (cpg) {
            case 8: return launch(k_w4a16_gemv_m8<8, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>, packed, a, p, st);
            case 4: return launch(k_w4a16_gemv_m8<4, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>, packed, a, p, st);
            case 2: return launch(k_w4a16_gemv_m8<2, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>, packed, a, p, st);
            default: return launch(k_w4a16_gemv_m8<1, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>, packed, a, p, st);
        }
    }
    switch (cpg) {
        case 8: return launch(k_w4a16_gemv_m16<8, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>, packed, a, p, st);
        case 4: return launch(k_w4a16_gemv_m16<4, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>, packed, a, p, st);
        case 2: return launch(k_w4a16_gemv_m16<2, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>, packed, a, p, st);
        default: return launch(k_w4a16_gemv_m16<1, ASYM, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>, packed, a, p, st);
    }
}

// W4A16 decode launch for one K-split case (all group sizes and widths).
// The token tile (8 or 16) follows a.M, or the per-group bound when grouped.
// SB: bf16 parameters; asymmetric when a.offs_b is set.  F32: fp32 outputs
// a.y32 without bias.
template <bool SPLIT, bool SWIGLU = false, bool GROUPED = false, bool SB = false,
          bool F32 = false, bool Q8 = false>
int launch_w4a16_variant(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                         cudaStream_t st) {
    const int gq = a.G / 32;
    const int cpg = (gq % 8 == 0) ? 8 : (gq % 4 == 0) ? 4 : (gq % 2 == 0) ? 2 : 1;
    const bool asym = SB ? a.offs_b != nullptr : a.zeros != nullptr;
    if ((GROUPED ? a.gmax : a.M) <= 8)
        return asym ? launch_w4a16_cpg<1, true, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>(cpg, packed, a, p, st)
                    : launch_w4a16_cpg<1, false, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>(cpg, packed, a, p, st);
    return asym ? launch_w4a16_cpg<2, true, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>(cpg, packed, a, p, st)
                : launch_w4a16_cpg<2, false, SPLIT, SWIGLU, GROUPED, SB, F32, Q8>(cpg, packed, a, p, st);
}

}  // namespace
}  // namespace w4
