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
// D[weight rows x BN tokens] (fp32, TMEM) += W_hat[rows x 64] * x[BN x 64]^T
// per 64-column stage; W_hat = s (code - z) is rounded once to bf16.  Tiles:
//   one CTA   128 weight rows x BN tokens (BN 256 or 128), tcgen05.mma
//             cta_group::1, M = 128;
//   CTA pair  256 weight rows x 256 tokens on a cluster of two CTAs: each
//             CTA stages 128 of the tokens (its half of the B operand) and
//             dequantizes its 128 rows (its half of A); rank 0 issues
//             tcgen05.mma cta_group::2 with M = 256, N = 256, and each CTA's
//             TMEM receives its 128 rows x 256 tokens.
// A unit of work is (output tile, K slice).  When a plan splits K S ways,
// each unit writes its fp32 partial tile to the workspace and takes a
// ticket; the last of the tile's S units to arrive adds the partials in
// split order 0..S-1 (its own term straight from TMEM), so every output is
// summed in the same order on every run and no unit ever waits for another.
//
// Warp roles (96 + 256 DQG + 128 threads, one CTA per SM, persistent):
//   warp 0      TMA of the x tile (128-byte swizzle) into an NST-stage ring,
//               released by the MMAs
//   warp 1      TMEM allocation (2 BN columns: two accumulators); one thread
//               issues the MMAs (4 x K=16 per stage)
//   warp 2      TMA of the packed tile (128 rows x 32 bytes) into an
//               NSP-stage ring, released by the dequantizing warps
//   next 8 DQG  dequantize into the 128-byte-swizzled K-major bf16 A ring
//               (NSA stages): DQG groups of 8 warps take turns stage by
//               stage, one weight row and 32 columns per thread
//   last 4      epilogue: tcgen05.ld of the accumulator, + bias, bf16 stores
//               (or fp32 stores without bias for a row-parallel shard's
//               partial sums; or the split-K hand-off)
// Every mbarrier and counter wait is bounded; a failed wait raises the CTA
// abort flag and the device error flag, in-flight copies and MMAs are
// drained before exit.
#include "w4_device.cuh"
#include "w4_internal.h"

#include <cstdlib>

namespace w4 {
namespace {

constexpr int BM = 128;                 // weight rows per tile (MMA M)
constexpr int BK = 64;                  // columns per K block (one 128-byte swizzle row)
constexpr int P_BYTES = BM * BK / 2;    // 4 KB of packed codes per K block
constexpr int A_BYTES = BM * BK * 2;    // 16 KB of bf16 A per K block
constexpr int DQ_GROUP_THREADS = 256;   // dequantizing threads per stage
constexpr int DQ_TPR = DQ_GROUP_THREADS / BM;  // threads per weight row
constexpr int EPI_THREADS = 128;
constexpr int DQ_BASE = 96;             // first dequantizing thread (after 3 role warps)

// DQG groups of DQ_GROUP_THREADS dequantizing threads
template <int DQG>
__host__ __device__ constexpr int threads_of() { return DQ_BASE + DQG * DQ_GROUP_THREADS + EPI_THREADS; }

struct GemmArgs {
    const float* scales;
    const uint8_t* zeros;
    const uint16_t* scales_b;   // bf16 parameter layout (SB): scales, and
    const uint16_t* offs_b;     // offsets (8 - z) s for asymmetric groups
    const float* bias;
    uint16_t* y;
    float* y32;         // fp32 outputs without bias instead of y (row-parallel partials)
    float* partial;     // S > 1: [ntiles, S, CTAs per tile, BN tokens, 128 rows] fp32
    int* tickets;       // [ntiles] when S > 1
    int* err;
    int M, N, K, G, Ng;
    int nks;        // k stages over K
    int TB;         // token blocks
    int ntiles;
    int S, spl;     // K splits, stages per split
    int units;      // ntiles * S
    // grouped launches (experts): x [T = M, K] rows sorted by group, goff[E+1]
    // token offsets on the device, weights / scales / bias stacked [E * Ne, ...],
    // y [T, Ne]; NBg row blocks per group
    const int* goff;
    int E, Ne, NBg;
};

template <int NST, int NSA, int NSP>
struct Ctl {
    uint64_t tfull[NST], tempty[NST];
    uint64_t pfull[NSP], pempty[NSP];
    uint64_t afull[NSA], aempty[NSA];
    uint64_t accfull[2], accempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int last;   // the tile's splits are all written (split-K hand-off)
};

// KB: K blocks of 64 columns per stage
template <int XR, int NST, int NSA, int NSP, int KB>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)NST * XR * BK * KB * 2 + (size_t)NSA * A_BYTES * KB +
           (size_t)NSP * P_BYTES * KB +
           (sizeof(Ctl<NST, NSA, NSP>) + 15) / 16 * 16;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    const uint32_t s = smem_u32(p);
    return p + (((s + 1023u) & ~1023u) - s);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One unit of work: output tile `tile` (split s, stages [ks0, ks1)), the
// weight rows gbase + nloc0 .. (of which the first nlim are the layer's),
// the token rows [t0, tend).
struct Unit {
    int tile, s, ks0, ks1;
    int gbase;     // first weight row of the unit's matrix (group e: e * Ne)
    int nloc0;     // first row of the tile inside that matrix (= y column)
    int nlim;      // rows of the matrix (N, or Ne when grouped) = y row stride
    int t0, tend;  // token rows of x and y
};

// GRP: a grouped launch; gpre[e] is the number of token tiles of the groups
// before e (gpre[E] = all tiles), units are (tile item, row block).
template <bool GRP, int BN, int RB>
__device__ __forceinline__ Unit unit_of(const GemmArgs& a, int u, const int* gpre) {
    Unit w;
    if constexpr (GRP) {
        const int item = u / a.NBg, nb = u - item * a.NBg;
        int lo = 0, hi = a.E - 1;                    // the group whose tiles hold item
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (gpre[mid] <= item) lo = mid; else hi = mid - 1;
        }
        const int o0 = __ldg(a.goff + lo), o1 = __ldg(a.goff + lo + 1);
        w.tile = u; w.s = 0; w.ks0 = 0; w.ks1 = a.nks;
        w.gbase = lo * a.Ne; w.nloc0 = nb * RB; w.nlim = a.Ne;
        w.t0 = o0 + (item - gpre[lo]) * BN;
        w.tend = min(o1, w.t0 + BN);
    } else {
        w.tile = u / a.S;
        w.s = u - w.tile * a.S;
        const int nb = w.tile / a.TB, tb = w.tile - nb * a.TB;
        w.ks0 = w.s * a.spl;
        w.ks1 = min(w.ks0 + a.spl, a.nks);
        w.gbase = 0; w.nloc0 = nb * RB; w.nlim = a.N;
        w.t0 = tb * BN; w.tend = a.M;
    }
    return w;
}

// SB: bf16 parameters; the dequantized weight is s (code - 8) + o.
// GRP: a grouped linear over E groups (experts), the grouped matmul of "Yeniden
// paketlenmiş QAT Gemma 4 26B-A4B, tek bir TPU v6e'de FP8 işlemenin 1.9 katı
// verimle sunuluyor", section "vLLM'in TPU backend'inde değişen ne oldu", for
// groups of many tokens: group e's tokens, rows goff[e] .. goff[e+1] - 1 of x,
// times its own Ne x K matrix, in tiles of BN tokens.  Before the role split
// warp 2 validates the offsets and writes the tiles' prefix sum to shared
// memory; every role then maps a unit to (group, token tile, row block).  A
// tile's rows past its group are computed but not stored.  No K split.
template <int BN, int NST, int NSA, int NSP, int DQG, bool PAIR, int KB, bool SB = false,
          bool GRP = false>
__global__ void __launch_bounds__(threads_of<DQG>(), 1)
k_w4a16_gemm_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmP,
                const GemmArgs a) {
    static_assert(!(GRP && PAIR), "grouped tiles run on single CTAs");
    constexpr int THREADS = threads_of<DQG>();
    constexpr int XR = PAIR ? BN / 2 : BN;                  // x rows staged by this CTA
    constexpr int RB = PAIR ? 2 * BM : BM;                  // weight rows per tile
    constexpr int SK = BK * KB;                             // columns per stage
    constexpr int X_BYTES = XR * SK * 2;                    // KB blocks of XR x 128 B
    constexpr int A_ST = A_BYTES * KB, P_ST = P_BYTES * KB; // A / packed bytes per stage
    constexpr int DQ_COLS = SK / DQ_TPR;                    // columns per thread per stage
    constexpr int DQ_CHUNKS = DQ_COLS / 8;                  // 16-byte bf16 chunks per thread
    constexpr uint32_t TMEM_COLS = 2 * BN;
    constexpr uint32_t IDESC = idesc_bf16_f32(RB, BN);
    constexpr int NCTA = PAIR ? 2 : 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = align1024(smem_raw);
    uint8_t* xs = base;                                     // NST x X_BYTES
    uint8_t* as = xs + NST * X_BYTES;                       // NSA x A_ST
    uint8_t* ps = as + NSA * A_ST;                          // NSP x P_ST
    auto* ctl = reinterpret_cast<Ctl<NST, NSA, NSP>*>(ps + NSP * P_ST);
    // grouped: tiles before each group, E + 1 ints after the control block
    int* gpre = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ctl) +
                                       (sizeof(Ctl<NST, NSA, NSP>) + 15) / 16 * 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a pair tile is worked on by the two CTAs of a cluster: rank 0 issues
    // the MMAs, each CTA stages its half of x and dequantizes its 128 rows
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const int slot = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int nslots = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    // shared::cluster address of a barrier in the rank-0 CTA
    auto at_rank0 = [&](uint64_t* bar) { return mapa_shared(smem_u32(bar), 0); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) { mbar_init(&ctl->tfull[i], 1); mbar_init(&ctl->tempty[i], 1); }
        for (int i = 0; i < NSP; ++i) {
            mbar_init(&ctl->pfull[i], 1);
            mbar_init(&ctl->pempty[i], DQ_GROUP_THREADS / 32);
        }
        for (int i = 0; i < NSA; ++i) {
            mbar_init(&ctl->afull[i], NCTA * DQ_GROUP_THREADS / 32);
            mbar_init(&ctl->aempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->accfull[i], 1);
            mbar_init(&ctl->accempty[i], NCTA * EPI_THREADS / 32);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        ctl->last = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) { tma_prefetch_desc(&tmX); tma_prefetch_desc(&tmP); }
    if constexpr (GRP) {
        if (warp == 2) {
            // group e has ceil(count / BN) token tiles; offsets outside [0, T]
            // or decreasing leave the group out and raise W4_ERR_GROUP_TOKENS
            int run = 0;
            if (lane == 0) gpre[0] = 0;
            for (int e0 = 0; e0 < a.E; e0 += 32) {
                const int e = e0 + lane;
                int n = 0;
                if (e < a.E) {
                    const int o0 = __ldg(a.goff + e), o1 = __ldg(a.goff + e + 1);
                    const bool ok = o0 >= 0 && o1 >= o0 && o1 <= a.M;
                    if (!ok) atomicCAS(a.err, 0, W4_ERR_GROUP_TOKENS);
                    n = ok ? (o1 - o0 + BN - 1) / BN : 0;
                }
                int v = n;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int t = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += t;
                }
                if (e < a.E) gpre[e + 1] = run + v;
                run += __shfl_sync(0xffffffffu, v, 31);
            }
            // offsets valid one by one can still overlap and list more tiles
            // than T tokens need; every access stays in bounds, but flag it
            if (lane == 0 && run > a.E + (a.M + BN - 1) / BN) atomicCAS(a.err, 0, W4_ERR_GROUP_TOKENS);
        }
    }
    if constexpr (PAIR) {
        if (warp == 1) { tmem_alloc_pair(&ctl->tmem_base, TMEM_COLS); tmem_relinquish_pair(); }
        tc_fence_before();
        cluster_sync();             // both CTAs' barriers exist before any remote arrival
    } else {
        if (warp == 1) { tmem_alloc(&ctl->tmem_base, TMEM_COLS); tmem_relinquish(); }
        tc_fence_before();
        __syncthreads();
    }
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int units = GRP ? gpre[a.E] * a.NBg : a.units;

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ TMA
        // warp 0 loads the x tiles (NST-stage ring, released by the MMAs),
        // warp 2 the packed weight tiles (NSP-stage ring, released by the
        // dequantizing threads once they hold the bytes in registers)
        if (lane == 0) {
            const bool is_x = warp == 0;
            const int ring = is_x ? NST : NSP;
            uint64_t* full = is_x ? ctl->tfull : ctl->pfull;
            uint64_t* empty = is_x ? ctl->tempty : ctl->pempty;
            const uint64_t pol = is_x ? policy_evict_last() : policy_evict_first();
            uint32_t it = 0;
            bool ok = true;
            for (int u = slot; u < units && ok; u += nslots) {
                const Unit w = unit_of<GRP, BN, RB>(a, u, gpre);
                const int ks0 = w.ks0, ks1 = w.ks1;
                for (int ks = ks0; ks < ks1; ++ks, ++it) {
                    const int st = it % ring;
                    if (it >= (uint32_t)ring &&
                        !mbar_wait(&empty[st], ((it / ring) & 1) ^ 1, &ctl->abort, a.err)) {
                        ok = false;
                        break;
                    }
                    if (is_x) {
                        if constexpr (PAIR) {
                            // both halves land on the rank-0 barrier
                            if (rank == 0) mbar_arrive_expect_tx(&full[st], 2 * X_BYTES);
                            for (int kb = 0; kb < KB; ++kb)
                                tma_load_2d_pair(xs + st * X_BYTES + kb * XR * 128, &tmX, ks * SK + kb * BK,
                                                 w.t0 + (int)rank * XR, at_rank0(&full[st]), pol);
                        } else {
                            mbar_arrive_expect_tx(&full[st], X_BYTES);
                            for (int kb = 0; kb < KB; ++kb)
                                tma_load_2d(xs + st * X_BYTES + kb * XR * 128, &tmX, ks * SK + kb * BK,
                                            w.t0, &full[st], pol);
                        }
                    } else {
                        mbar_arrive_expect_tx(&full[st], P_ST);
                        tma_load_2d(ps + st * P_ST, &tmP, ks * (SK / 2),
                                    w.gbase + w.nloc0 + (int)rank * BM, &full[st], pol);
                    }
                }
            }
            // (the x copies of rank 1 complete on the rank-0 barrier, which
            // rank 0 drains; the pair leaves together through cluster_sync)
            if ((!ok || ctl->abort) && (!PAIR || !is_x || rank == 0)) {
                const uint32_t first = it > (uint32_t)ring ? it - ring : 0;
                for (uint32_t j = first; j < it; ++j)
                    mbar_wait_drain(&full[j % ring], (j / ring) & 1, a.err);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && rank == 0) {
            // waits on barriers that the other CTA of a pair also arrives on
            auto wait = [&](uint64_t* bar, uint32_t parity) {
                if constexpr (PAIR) return mbar_wait_cluster(bar, parity, &ctl->abort, a.err);
                else return mbar_wait(bar, parity, &ctl->abort, a.err);
            };
            uint32_t it = 0, ia = 0, tc = 0;
            bool ok = true;
            for (int u = slot; u < units && ok; u += nslots, ++tc) {
                const Unit w = unit_of<GRP, BN, RB>(a, u, gpre);
                const int ks0 = w.ks0, ks1 = w.ks1;
                const uint32_t b = tc & 1;
                if (tc >= 2 && !wait(&ctl->accempty[b], ((tc / 2) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + b * BN;
                for (int ks = ks0; ks < ks1; ++ks, ++it, ++ia) {
                    const int st = it % NST, sa = ia % NSA;
                    if (!wait(&ctl->tfull[st], (it / NST) & 1) || !wait(&ctl->afull[sa], (ia / NSA) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(as + sa * A_ST);
                    const uint32_t x_addr = smem_u32(xs + st * X_BYTES);
                    // K step i: block i / 4 (A_BYTES / XR x 128 B apart), 32 B per step inside it
                    auto a_k = [&](int i) { return a_addr + (i >> 2) * A_BYTES + 32 * (i & 3); };
                    auto x_k = [&](int i) { return x_addr + (i >> 2) * (XR * 128) + 32 * (i & 3); };
                    if constexpr (PAIR) {
#pragma unroll
                        for (int i = 0; i < SK / 16; ++i)
                            tc_mma_f16_pair(d, smem_desc_sw128(a_k(i)), smem_desc_sw128(x_k(i)), IDESC,
                                            (ks > ks0 || i > 0) ? 1u : 0u);
                        tc_commit_pair(&ctl->tempty[st], 3);
                        tc_commit_pair(&ctl->aempty[sa], 3);
                    } else {
#pragma unroll
                        for (int i = 0; i < SK / 16; ++i)
                            tc_mma_f16(d, smem_desc_sw128(a_k(i)), smem_desc_sw128(x_k(i)), IDESC,
                                       (ks > ks0 || i > 0) ? 1u : 0u);
                        tc_commit(&ctl->tempty[st]);
                        tc_commit(&ctl->aempty[sa]);
                    }
                }
                if (!ok) break;
                if constexpr (PAIR) tc_commit_pair(&ctl->accfull[b], 3);
                else tc_commit(&ctl->accfull[b]);
            }
            // every MMA issued by this thread completes before the CTA ends
            if constexpr (PAIR) tc_commit_pair(&ctl->drain, 1);
            else tc_commit(&ctl->drain);
            mbar_wait_drain(&ctl->drain, 0, a.err);
        }
    } else if (threadIdx.x < DQ_BASE + DQG * DQ_GROUP_THREADS) {
        // ------------------------------------------------------------ dequantize
        // DQ_GROUPS groups take turns stage by stage, so that several stages
        // are dequantized at once.  In a group, thread (r, h) converts weight
        // row r, columns [DQ_COLS h, DQ_COLS h + DQ_COLS) of the stage; the
        // threads of a row are neighbouring lanes, so a warp reads one
        // contiguous span of the packed tile.
        constexpr int DQ_GROUPS = DQG;
        static_assert(NSP % DQ_GROUPS == 0 && NSA >= 2, "stage rings vs dequant groups");
        const int dt = threadIdx.x - DQ_BASE;
        const int grp = dt / DQ_GROUP_THREADS, gt = dt % DQ_GROUP_THREADS;
        const int r = gt / DQ_TPR, h = gt % DQ_TPR;
        uint32_t it = 0;
        for (int u = slot; u < units; u += nslots) {
            const Unit w = unit_of<GRP, BN, RB>(a, u, gpre);
            const int ks0 = w.ks0, ks1 = w.ks1;
            // first stage of this unit that falls to this group
            const int lead = (int)((grp - it % DQ_GROUPS + DQ_GROUPS) % DQ_GROUPS);
            it += (uint32_t)lead;
            const int n = w.gbase + min(w.nloc0 + (int)rank * BM + r, w.nlim - 1);
            const float* srow = a.scales + (size_t)n * a.Ng;
            const uint8_t* zrow = a.zeros ? a.zeros + (size_t)n * a.Ng : nullptr;
            const uint16_t* sbrow = SB ? a.scales_b + (size_t)n * a.Ng : nullptr;
            const uint16_t* obrow = SB && a.offs_b ? a.offs_b + (size_t)n * a.Ng : nullptr;
            // scale and zero point (SB: bf16 scale and offset) of this
            // thread's columns, loaded one turn ahead
            auto group_of = [&](int ks) { return min((ks * SK + DQ_COLS * h) / a.G, a.Ng - 1); };
            auto scale_at = [&](int g) -> float {
                return SB ? __uint_as_float((uint32_t)__ldg(sbrow + g) << 16) : __ldg(srow + g);
            };
            auto zero_at = [&](int g) -> float {
                if constexpr (SB) return obrow ? __uint_as_float((uint32_t)__ldg(obrow + g) << 16) : 0.f;
                else return zrow ? (float)__ldg(zrow + g) : 8.f;
            };
            const int kf = min(ks0 + lead, ks1 - 1);
            float sc = scale_at(group_of(kf));
            float zz = zero_at(group_of(kf));
            int ks = ks0 + lead;
            for (; ks < ks1; ks += DQ_GROUPS, it += DQ_GROUPS) {
                const int sp = it % NSP, sa = it % NSA;
                float nsc = sc, nzz = zz;
                if (ks + DQ_GROUPS < ks1) {
                    const int g = group_of(ks + DQ_GROUPS);
                    nsc = scale_at(g);
                    nzz = zero_at(g);
                }
                // (128 + c) s + cc: cc = -(128 + z) s, or with an offset o - 136 s
                const float cc = SB ? fmaf(-136.f, sc, zz) : -(128.f + zz) * sc;
                // one arrival per warp on pempty / afull (after __syncwarp),
                // so a stage costs 2 x 8 barrier updates, not 2 x 256
                bool ok = __all_sync(0xffffffffu,
                                     mbar_wait(&ctl->pfull[sp], (it / NSP) & 1, &ctl->abort, a.err));
                uint32_t wv[DQ_CHUNKS];
                if (ok) {
                    const uint8_t* prow = ps + sp * P_ST + r * (SK / 2) + h * (DQ_COLS / 2);
                    if constexpr (DQ_CHUNKS >= 4) {
#pragma unroll
                        for (int i = 0; i < DQ_CHUNKS / 4; ++i) {
                            const uint4 q = *reinterpret_cast<const uint4*>(prow + 16 * i);
                            wv[4 * i] = q.x; wv[4 * i + 1] = q.y; wv[4 * i + 2] = q.z; wv[4 * i + 3] = q.w;
                        }
                    } else {
                        const uint2 q = *reinterpret_cast<const uint2*>(prow);
                        wv[0] = q.x; wv[1] = q.y;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->pempty[sp]);
                }
                if (ok && it >= (uint32_t)NSA)
                    ok = mbar_wait(&ctl->aempty[sa], ((it / NSA) & 1) ^ 1, &ctl->abort, a.err);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    uint8_t* arow = as + sa * A_ST + r * 128;
                    // With two K blocks a stage, the two threads of a row (h = 0, 1:
                    // neighbouring lanes) write one chunk each of blocks 0 and 1; in
                    // the same swizzled position they would hit the same banks, so
                    // h = 1 takes its chunks in the order jj ^ 4 (a select between
                    // two register indices, no dynamic indexing)
                    constexpr int HX = DQ_CHUNKS == 8 ? 4 : 0;
#pragma unroll
                    for (int jj = 0; jj < DQ_CHUNKS; ++jj) {
                        const int lc = h ? (jj ^ HX) : jj;      // this thread's chunk
                        const int jg = DQ_CHUNKS * h + lc;      // 16-byte chunk of the stage's row
                        const int j = jg & 7;                   // chunk inside its K block
                        const uint32_t w = h ? wv[jj ^ HX] : wv[jj], wh = w >> 4;
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
                        *reinterpret_cast<uint4*>(arow + (jg >> 3) * A_BYTES + ((j ^ (r & 7)) << 4)) = o;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR) mbar_arrive_cluster(at_rank0(&ctl->afull[sa]));
                        else mbar_arrive(&ctl->afull[sa]);
                    }
                }
                sc = nsc;
                zz = nzz;
            }
            // `it` now points past this unit by less than DQ_GROUPS stages
            it -= (uint32_t)(ks - ks1);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                            // TMEM lane quarter of this warp
        const int r = q * 32 + lane;
        const int etid = threadIdx.x - (THREADS - EPI_THREADS);
        uint32_t tc = 0;
        for (int u = slot; u < units; u += nslots, ++tc) {
            const Unit w = unit_of<GRP, BN, RB>(a, u, gpre);
            const int tile = w.tile, s = w.s;
            const uint32_t b = tc & 1;
            // the same outcome for all 128 epilogue threads, which then take
            // the same branch (aligned tcgen05.ld, named barriers)
            bool ok = named_bar_and(2, EPI_THREADS,
                                    mbar_wait(&ctl->accfull[b], (tc / 2) & 1, &ctl->abort, a.err));
            tc_fence_after();
            const int n = w.nloc0 + (int)rank * BM + r;        // output column
            const int NO = w.nlim, TE = w.tend;                 // y row stride, token limit
            int* ticket = a.tickets + (size_t)tile * NCTA + rank;   // per 128-row half
            const float bn = (a.bias && n < NO) ? __ldg(a.bias + w.gbase + n) : 0.f;
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN;
            const int t0 = w.t0;
            if (ok && a.S == 1) {
                for (int j = 0; j < BN / 32 && t0 + j * 32 < TE; ++j) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tacc + j * 32, v);
                    tc_wait_ld();
                    if (n < NO) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int t = t0 + j * 32 + i;
                            if (t < TE) {
                                if (a.y32) a.y32[(size_t)t * NO + n] = __uint_as_float(v[i]);
                                else a.y[(size_t)t * NO + n] = f32_to_bf16_bits(__uint_as_float(v[i]) + bn);
                            }
                        }
                    }
                }
            } else if (ok) {
                // 1. this split's fp32 partial tile into the workspace: one
                //    contiguous region per (tile, split, CTA), token-major
                //    with the 128 rows innermost, so that every warp store
                //    (and every load of the reduction) covers 32 consecutive
                //    floats.  (A layout with each thread's 32 tokens
                //    contiguous, stored as 16-byte words at a 128-byte stride
                //    across the warp, gave wrong accumulators in the CTA's
                //    later units in the parity tests; see the design notes.)
                float* ptile = a.partial + (((size_t)tile * a.S) * NCTA + rank) * (BM * BN);
                const size_t split_stride = (size_t)NCTA * BM * BN;     // floats between splits
                for (int j = 0; j < BN / 32 && t0 + j * 32 < TE; ++j) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tacc + j * 32, v);
                    float* dst = ptile + s * split_stride + (size_t)j * (BM * 32) + r;
#pragma unroll
                    for (int i = 0; i < 32; ++i) dst[(size_t)i * BM] = __uint_as_float(v[i]);
                }
                // 2. publish it and take a ticket; the last of the S splits
                //    to arrive reduces the whole tile, so no split ever waits
                //    for another (nothing depends on the S units being
                //    resident at the same time)
                named_bar_sync(2, EPI_THREADS);
                if (etid == 0) ctl->last = atom_add_acq_rel_gpu(ticket, 1) == a.S - 1;
                named_bar_sync(2, EPI_THREADS);
                if (ctl->last) {
                    // 3. partials added in split order 0..S-1 (this split's own
                    //    term straight from TMEM), the same order whichever
                    //    split arrives last; the 32 loads of a block are
                    //    independent, so they are in flight together
                    for (int j = 0; j < BN / 32 && t0 + j * 32 < TE; ++j) {
                        float acc[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) acc[i] = 0.f;
                        for (int qq = 0; qq < a.S; ++qq) {
                            uint32_t v[32];
                            if (qq == s) {
                                tmem_ld_32x32b_x32(tacc + j * 32, v);
                            } else {
                                const float* src = ptile + qq * split_stride + (size_t)j * (BM * 32) + r;
#pragma unroll
                                for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(ld_cg_f32(src + (size_t)i * BM));
                            }
#pragma unroll
                            for (int i = 0; i < 32; ++i) acc[i] += __uint_as_float(v[i]);
                        }
                        if (n < NO) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int t = t0 + j * 32 + i;
                                if (t < TE) {
                                    if (a.y32) a.y32[(size_t)t * NO + n] = acc[i];
                                    else a.y[(size_t)t * NO + n] = f32_to_bf16_bits(acc[i] + bn);
                                }
                            }
                        }
                    }
                    // 4. every split has taken its ticket: reset the counter
                    if (etid == 0) *ticket = 0;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_cluster(at_rank0(&ctl->accempty[b]));
                else mbar_arrive(&ctl->accempty[b]);
            }
        }
    }

    tc_fence_before();
    if constexpr (PAIR) cluster_sync();     // no CTA leaves while its peer may still use it
    else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int BN, int NST, int NSA, int NSP, int DQG, bool PAIR, int KB, bool SB = false,
          bool GRP = false>
struct Variant {
    static constexpr int XR = PAIR ? BN / 2 : BN;
    static constexpr size_t smem = smem_bytes<XR, NST, NSA, NSP, KB>();
    static constexpr size_t kSmemMax = 232448;
    static_assert(smem <= kSmemMax, "shared memory");
    static constexpr auto kernel = k_w4a16_gemm_tc<BN, NST, NSA, NSP, DQG, PAIR, KB, SB, GRP>;
    // grouped: the largest group count whose tile prefix sum fits
    static constexpr int kMaxGroups = (int)((kSmemMax - smem) / 4) - 1;

    static bool prepare() {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)(GRP ? kSmemMax : smem)) == cudaSuccess;
    }

    static cudaLaunchConfig_t config(int grid, cudaStream_t stream, cudaLaunchAttribute* at) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3((unsigned)threads_of<DQG>());
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = PAIR ? 2 : 1;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = PAIR ? 1 : 0;
        return cfg;
    }

    // CTAs (or CTA pairs) of this variant resident at once on this device:
    // the persistent grid is at most this
    static int slots(int sm_count) {
        static int cache[64] = {0};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
        if (cache[dev] == 0) {
            int n = 0;
            if (prepare()) {
                if (PAIR) {
                    cudaLaunchAttribute at[1];
                    cudaLaunchConfig_t cfg = config(2 * sm_count, nullptr, at);
                    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
                } else {
                    int per_sm = 0;
                    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads_of<DQG>(),
                                                                      smem) == cudaSuccess)
                        n = per_sm * sm_count;
                }
            }
            cudaGetLastError();
            cache[dev] = n > 0 ? n : -1;
        }
        return cache[dev] > 0 ? cache[dev] : 0;
    }

    static int launch(const uint16_t* x, const uint8_t* packed, const GemmPlan& p, GemmArgs& a,
                      int Kp, cudaStream_t stream) {
        CUtensorMap tmX, tmP;
        if (!encode_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)a.K, (uint64_t)a.M,
                            (uint64_t)a.K * 2, BK, XR, CU_TENSOR_MAP_SWIZZLE_128B))
            return W4_ERR_CUDA;
        if (!encode_tmap_2d(&tmP, CU_TENSOR_MAP_DATA_TYPE_UINT8, packed, (uint64_t)(Kp / 2),
                            (uint64_t)a.N, (uint64_t)(Kp / 2), BK * KB / 2, BM, CU_TENSOR_MAP_SWIZZLE_NONE))
            return W4_ERR_CUDA;
        if (!prepare()) return W4_ERR_CUDA;
        cudaLaunchAttribute at[1];
        cudaLaunchConfig_t cfg = config(p.grid, stream, at);
        if (GRP) cfg.dynamicSmemBytes = smem + ((size_t)(a.E + 1) * 4 + 15) / 16 * 16;
        if (cudaLaunchKernelEx(&cfg, kernel, tmX, tmP, a) != cudaSuccess) return W4_ERR_CUDA;
        return W4_OK;
    }

    // A grouped launch: x [T, K] rows sorted by group, the E groups' Ne x K
    // matrices stacked (the tensor map covers E * Ne rows), no K split.
    static int launch_grouped(const uint16_t* x, const int* goff, const uint8_t* packed,
                              const float* scales, const uint8_t* zeros, const float* bias,
                              uint16_t* y, int T, int E, int Ne, int K, int Kp, int G, int* err,
                              int sm_count, cudaStream_t stream) {
        if (E > kMaxGroups) return W4_ERR_UNSUPPORTED_SHAPE;
        GemmArgs a{};
        a.scales = scales; a.zeros = zeros; a.bias = bias; a.y = y; a.err = err;
        a.goff = goff; a.E = E; a.Ne = Ne; a.NBg = (Ne + BM - 1) / BM;
        a.M = T; a.N = E * Ne; a.K = K; a.G = G; a.Ng = Kp / G;
        a.nks = (K + BK * KB - 1) / (BK * KB);
        a.S = 1; a.spl = a.nks; a.TB = 1;
        GemmPlan p;
        const long long ub = ((long long)E + (T + BN - 1) / BN) * a.NBg;   // units at most
        const int sl = slots(sm_count);
        if (sl < 1) return W4_ERR_CUDA;
        p.grid = (int)(ub < sl ? ub : sl);
        if (p.grid < 1) return W4_OK;
        return launch(x, packed, p, a, Kp, stream);
    }
};

using Single256 = Variant<256, 4, 4, 8, 1, false, 1>;
using Single128 = Variant<128, 8, 4, 8, 1, false, 1>;
using Pair256 = Variant<256, 6, 4, 8, 1, true, 1>;
using Single256B = Variant<256, 4, 4, 8, 1, false, 1, true>;
using Single128B = Variant<128, 8, 4, 8, 1, false, 1, true>;
using Pair256B = Variant<256, 6, 4, 8, 1, true, 1, true>;
// 128 columns per stage (two K blocks): half the per-stage hand-offs for the
// same MMA work; group sizes that are multiples of 64 only (a dequantizing
// thread's 64 columns must lie in one group)
using Single256K2 = Variant<256, 2, 2, 4, 1, false, 2>;
// 64-token tiles for small and mid-range M (17 .. ~128 tokens) and expert
// groups of a few dozen tokens: the MMA is 1/4 of a 256-token stage, so the
// dequantized A ring is deeper to keep several stages in flight
using Single64K2 = Variant<64, 4, 3, 6, 1, false, 2>;
using Single64 = Variant<64, 8, 6, 12, 1, false, 1>;
using Single64K2B = Variant<64, 4, 3, 6, 1, false, 2, true>;
using Single64B = Variant<64, 8, 6, 12, 1, false, 1, true>;
using Pair256K2 = Variant<256, 4, 2, 4, 1, true, 2>;
// grouped (experts) launches: 64- and 256-token tiles
using Grp64K2 = Variant<64, 4, 3, 6, 1, false, 2, false, true>;
using Grp64 = Variant<64, 8, 6, 12, 1, false, 1, false, true>;
using Grp256K2 = Variant<256, 2, 2, 4, 1, false, 2, false, true>;
using Grp256 = Variant<256, 4, 4, 8, 1, false, 1, false, true>;
using Single256K2B = Variant<256, 2, 2, 4, 1, false, 2, true>;
using Pair256K2B = Variant<256, 4, 2, 4, 1, true, 2, true>;

}  // namespace

// Output tiles are 128 weight rows x BN tokens on one SM, or 256 rows x 256
// tokens on a CTA pair; K is split S ways when the tiles alone fill the GPU
// poorly.  Cost = waves x stages per unit x relative stage time, plus a
// charge per split for the fp32 partials and the hand-off.  A stage is bound
// by dequantizing its 128 rows at every tile width, so CTAs that share an SM
// share its rate: the stage time is multiplied by the CTAs per SM.
bool plan_gemm(int M, int N, int K, int G, int sm_count, GemmPlan* out) {
    if (M < 1 || N < 1 || K < 1 || sm_count < 1) return false;
    // W4_GEMM_BN (64, 128 or 256), W4_GEMM_SPLIT (1..8) and W4_GEMM_PAIR (0 or 1)
    // pin the plan (tuning sweeps, tests of every variant); read on every
    // call, which costs far less than one launch
    auto env_int = [](const char* name) {
        const char* e = std::getenv(name);
        return e ? std::atoi(e) : -1;
    };
    const int forced_bn = env_int("W4_GEMM_BN");
    const int forced_s = env_int("W4_GEMM_SPLIT");
    const int forced_pair = env_int("W4_GEMM_PAIR");
    struct Cand {
        bool pair;
        int BN;
        int kb;         // 64-column K blocks per stage
        int slots;      // CTAs (pairs) resident at once
        double stage;   // time of one stage, relative to one CTA's 128 x 256 x 64 stage
    };
    // measured on the 7B prefill shapes (gate_up M = 2048): a 128-column
    // stage takes 1.52 times a 64-column one (1.55 on a pair); a pair stage
    // (256 x 256 on two SMs) runs 1-3% slower than two single-CTA stages; a
    // 128-token stage takes as long as a 256-token one
    const int forced_kb = env_int("W4_GEMM_KB");
    // 64-token tiles: 0.96 of a 256-token stage (swept at M = 17 .. 2048 on
    // the 7B gate|up and down shapes)
    const Cand cands[7] = {
        {true, 256, 2, Pair256K2::slots(sm_count), 1.55},
        {false, 256, 2, Single256K2::slots(sm_count), 1.52},
        {true, 256, 1, Pair256::slots(sm_count), 1.02},
        {false, 256, 1, Single256::slots(sm_count), 1.0},
        {false, 128, 1, Single128::slots(sm_count), 1.0},
        {false, 64, 2, Single64K2::slots(sm_count), 1.46},
        {false, 64, 1, Single64::slots(sm_count), 0.96},
    };
    double best = 1e30;
    bool found = false;
    for (const Cand& c : cands) {
        if (c.slots < 1) continue;
        if (forced_pair == 0 && c.pair) continue;
        if (forced_pair == 1 && !c.pair) continue;
        if ((forced_bn == 64 || forced_bn == 128 || forced_bn == 256) && c.BN != forced_bn) continue;
        if ((forced_kb == 1 || forced_kb == 2) && c.kb != forced_kb) continue;
        if (c.kb == 2 && G % 64 != 0) continue;
        const int per_sm = std::max(1, (c.pair ? 2 * c.slots : c.slots) / sm_count);
        const double stage = c.stage * per_sm;
        const int nks = (K + BK * c.kb - 1) / (BK * c.kb);
        const int RB = c.pair ? 2 * BM : BM;
        const int TB = (M + c.BN - 1) / c.BN;
        const int ntiles = ((N + RB - 1) / RB) * TB;
        for (int S = 1; S <= 8 && S <= nks; ++S) {
            if (forced_s >= 1 && forced_s <= 8 && S != forced_s) continue;
            if (S > 1 && (long long)ntiles * (c.pair ? 2 : 1) > kMaxCounters) continue;
            const int spl = (nks + S - 1) / S;
            const int Se = (nks + spl - 1) / spl;
            if (Se != S) continue;
            const int units = ntiles * S;
            const int waves = (units + c.slots - 1) / c.slots;
            double cost = (double)waves * spl * stage;
            // split charge: each split writes its fp32 tile and the last one
            // to arrive reads the other S - 1 back
            if (S > 1) cost += 2.0 * waves * S * stage;
            if (cost < best * (1 - 1e-9)) {
                best = cost;
                found = true;
                GemmPlan p;
                p.pair = c.pair;
                p.kb = c.kb;
                p.BN = c.BN; p.TB = TB; p.ntiles = ntiles; p.S = S; p.spl = spl; p.nks = nks;
                p.units = units;
                p.grid = (c.pair ? 2 : 1) * (units < c.slots ? units : c.slots);
                p.ticket_bytes = S > 1 ? kCounterBytes : 0;
                // split partials: one 128-row x BN-token fp32 tile per split,
                // per CTA of each output tile
                p.ws_bytes = S > 1 ? p.ticket_bytes + (size_t)S * ntiles * (c.pair ? 2 : 1) *
                                                          BM * c.BN * 4
                                   : 0;
                *out = p;
            }
        }
    }
    return found;
}

int launch_w4a16_gemm(const uint16_t* x, const uint8_t* packed, const float* scales,
                      const uint8_t* zeros, const float* bias, uint16_t* y, int M, int N, int K,
                      int Kp, int G, const GemmPlan& p, void* workspace, int* err,
                      cudaStream_t stream, const uint16_t* scales_b, const uint16_t* offs_b,
                      float* y32) {
    GemmArgs a{};
    a.scales = scales; a.zeros = zeros; a.bias = bias; a.y = y; a.y32 = y32; a.err = err;
    a.scales_b = scales_b; a.offs_b = offs_b;
    a.M = M; a.N = N; a.K = K; a.G = G; a.Ng = Kp / G;
    a.nks = p.nks; a.TB = p.TB; a.ntiles = p.ntiles; a.S = p.S; a.spl = p.spl; a.units = p.units;
    if (p.S > 1) {
        a.tickets = static_cast<int*>(workspace);
        a.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + p.ticket_bytes);
    }
    if (p.BN == 64) {
        if (scales_b) return p.kb == 2 ? Single64K2B::launch(x, packed, p, a, Kp, stream)
                                       : Single64B::launch(x, packed, p, a, Kp, stream);
        return p.kb == 2 ? Single64K2::launch(x, packed, p, a, Kp, stream)
                         : Single64::launch(x, packed, p, a, Kp, stream);
    }
    if (scales_b) {
        if (p.kb == 2) {
            if (p.pair) return Pair256K2B::launch(x, packed, p, a, Kp, stream);
            return Single256K2B::launch(x, packed, p, a, Kp, stream);
        }
        if (p.pair) return Pair256B::launch(x, packed, p, a, Kp, stream);
        if (p.BN == 256) return Single256B::launch(x, packed, p, a, Kp, stream);
        return Single128B::launch(x, packed, p, a, Kp, stream);
    }
    if (p.kb == 2) {
        if (p.pair) return Pair256K2::launch(x, packed, p, a, Kp, stream);
        return Single256K2::launch(x, packed, p, a, Kp, stream);
    }
    if (p.pair) return Pair256::launch(x, packed, p, a, Kp, stream);
    if (p.BN == 256) return Single256::launch(x, packed, p, a, Kp, stream);
    return Single128::launch(x, packed, p, a, Kp, stream);
}

int launch_w4a16_grouped_gemm(const uint16_t* x, const int* goff, const uint8_t* packed,
                              const float* scales, const uint8_t* zeros, const float* bias,
                              uint16_t* y, int T, int E, int Ne, int K, int Kp, int G, int tile,
                              int* err, cudaStream_t stream) {
    const int sm = current_sm_count();
    const bool kb2 = G % 64 == 0;
    if (tile <= 64)
        return kb2 ? Grp64K2::launch_grouped(x, goff, packed, scales, zeros, bias, y, T, E, Ne, K,
                                             Kp, G, err, sm, stream)
                   : Grp64::launch_grouped(x, goff, packed, scales, zeros, bias, y, T, E, Ne, K, Kp,
                                           G, err, sm, stream);
    return kb2 ? Grp256K2::launch_grouped(x, goff, packed, scales, zeros, bias, y, T, E, Ne, K, Kp,
                                          G, err, sm, stream)
               : Grp256::launch_grouped(x, goff, packed, scales, zeros, bias, y, T, E, Ne, K, Kp, G,
                                        err, sm, stream);
}

}  // namespace w4
