// w4_internal.h - host-side declarations shared by the libw4 translation
// units (launchers, planning, device set-up).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/w4.h"

namespace w4 {

// ---------------------------------------------------------------- device
int current_sm_count();                 // SMs of the current device (cached)
int* device_error_flag();               // device address of the error flag
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t dim0, uint64_t dim1, uint64_t row_stride_bytes,
                    uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle);

// ---------------------------------------------------------------- decode
// Decode kernels (M <= 16): persistent CTAs of 8 consumer warps + 1 producer
// warp; a unit of work is (block of R output rows, slice of the padded K).
// A pipeline stage is 16 KB of packed weights: 128/R boxes of R rows x 128
// bytes (256 columns each), i.e. R rows x 32768/R columns.
// pipeline depth of the decode kernels' weight ring (16 KB stages); swept
// on the full bench: 3 beat 4 on the 7B step (3,748 vs 3,701 GB/s), the
// fused gate|up + SiLU at 8 tokens (19.1 vs 21.8 us) and the 12B shapes from
// 4 tokens, at 1-1.5% on the W4A8 GEMVs; 2, 6 and 8 were slower on the step
constexpr int kGemvStages = 3;
constexpr int kGemvStageBytes = 16384;
constexpr int kGemvConsumerWarps = 8;
constexpr int kGemvThreads = 32 * (kGemvConsumerWarps + 1);

struct GemvPlan {
    int R = 0;         // rows per unit (16, 32, 64 or 128)
    int SKE = 0;       // K columns per stage (32768 / R)
    int NB = 0;        // row blocks
    int nst = 0;       // stages over Kp
    int S = 0;         // K splits (global, combined by the last CTA)
    int spl = 0;       // stages per split
    int units = 0;     // NB * S
    int grid = 0;      // CTAs launched
    int cps = 0;       // CTAs per SM the plan is sized for
    int XS = 0;        // activation row stride in shared memory (bytes)
    int red = 0;       // bytes of the cross-warp reduction buffer
    size_t smem = 0;   // dynamic shared memory (bytes)
    size_t ws_bytes = 0;
    size_t list_off = 0;  // grouped plans: offset of the active-group list in shared memory
    bool f16 = false;  // W4A16: the fp16 inner loop (1-2 tokens, G >= 64), else bf16
    // K splits added inside a thread-block cluster: the S CTAs of a row block
    // form one cluster, ranks 1..S-1 store their partial sums into rank 0's
    // shared memory (a receive buffer at crecv_off), rank 0 adds them in
    // split order and writes y.  One unit per CTA; S <= 8.
    bool csplit = false;
    size_t crecv_off = 0;
};

// act_bytes: bytes per activation element (2 for bf16, 1 for int8).
// groups > 0: a grouped plan (one matrix of N rows per group, M = the token
// tile, N here = rows of all items expected): no K split, and room for a
// list of `groups` (group, token tile) items.
// Returns false if no plan fits (M too large).
bool plan_gemv(int M, int N, int Kp, int G, int act_bytes, int sm_count, GemvPlan* plan,
               int groups = 0);

struct GemvArgs {
    const void* x;            // bf16 [M, K] (W4A16) or int8 [M, Kp] (W4A8)
    const float* scales;      // [N, Ng] (W4A16) or [N] (W4A8)
    const uint8_t* zeros;     // [N, Ng] or nullptr
    const float* bias;        // [N] or nullptr
    const float* sx;          // [M] (W4A8)
    uint16_t* y;              // bf16 [M, N]
    int32_t* acc_out;         // [M, N] or nullptr (W4A8)
    void* partial;            // split-K partial sums [S, M, N]
    int* tickets;             // [NB] arrival counters
    int* err;                 // device error flag
    int M, N, K, Kp, G, Ng;
    int R, SKE, nst, S, spl, units, XS, red;
    int xtma;                 // activation rows are 16-byte aligned: stage them with TMA
    // grouped decode: x [M, K] rows sorted by group, goff[E+1] token offsets
    // of the E groups, weights/scales/zeros/bias stacked [E, N, ...], y [M, N];
    // groups are taken in tiles of at most gmax tokens
    const int* goff;
    int E, gmax, NBg;         // groups, token bound, row blocks per group
    int list_off;             // shared-memory offset of the (group, token tile) list
    int list_cap;             // its capacity in items
    // bf16 parameter layout (instead of scales / zeros): bf16 scales [N, Ng]
    // and, asymmetric, bf16 offsets (8 - z) s [N, Ng]
    const uint16_t* scales_b;
    const uint16_t* offs_b;
    // fp32 outputs [M, N] without bias (row-parallel partial sums), instead of y
    float* y32;
    // SwiGLU with INT8 outputs: qx [M, Fp] int8, sx_out [M], the CTA
    // arrival counter (the last counter of the workspace prefix; the one
    // before it holds the call generation)
    int8_t* qx;
    float* sx_out;
    int Fp;
    int* done;
    unsigned* ymax;           // [2][16] per-token max|y| (fp32 bits), by generation parity
    int csplit;               // K splits added in a cluster (GemvPlan::csplit)
    int coop;                 // INT8 outputs: ask for a cooperative launch (grid-wide hand-off)
    int pf;                   // stages of the first unit prefetched into L2 before the wait
    int xfirst;               // fp16 path: stages issued before holding for the staged activations (-1: no hold)
    int crecv_off;            // shared-memory offset of the cluster receive buffer
};

// The launchers encode the tensor map of `packed` for the plan's box shape
// and launch with programmatic dependent launch enabled.
// Whether decode CTAs copy their activation slice into shared memory with a
// bulk TMA copy (the bf16 path, which uses the slice as it is), instead of
// reading it from global memory while converting it (the fp16 path of 1-2
// tokens: measured 3.5% faster on the 7B step at one token).
// W4_GEMV_XTMA=0/1 overrides.
bool gemv_tma_activations(const GemvPlan& p);
// Decode with the SwiGLU epilogue: a.N = 2F paired gate/up rows, y [M, F].
int launch_w4a16_swiglu(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                        cudaStream_t stream);
// The same with the INT8 epilogue (a.qx, a.sx_out, a.Fp, a.done).
int launch_w4a16_swiglu_q8(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                           cudaStream_t stream);
int launch_w4a16_gemv_split(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                            cudaStream_t stream);
// Decode with the bf16 parameter layout (a.scales_b, a.offs_b).
int launch_w4a16_gemv_bf16p(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                            cudaStream_t stream);
// Grouped decode (MoE experts): the tensor map covers the E * N stacked rows.
int launch_w4a16_grouped(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                         cudaStream_t stream);
int launch_w4a16_gemv(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                      cudaStream_t stream);
// Decode with fp32 outputs a.y32 and no bias (split and unsplit plans).
int launch_w4a16_gemv_f32(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                          cudaStream_t stream);
int launch_w4a8_gemv(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                     cudaStream_t stream);
// Group-wise W4A8 (one weight scale per group of G columns, G < Kp):
// G = 32, 64, 128 or a multiple of 256.
bool w4a8_group_supported(int G);
int launch_w4a8g_gemv(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                      cudaStream_t stream);

// ---------------------------------------------------------------- prefill
// Tensor-core kernel for M > 16 (requires K % 8 == 0 and 16-byte aligned x).
// Split-K arrival counters occupy a fixed prefix of every workspace, so the
// partial sums of one call never land where another call's counters are.
constexpr size_t kCounterBytes = W4_WORKSPACE_COUNTER_BYTES;
constexpr int kMaxCounters = (int)(kCounterBytes / 4);

struct GemmPlan {
    bool pair = false; // CTA-pair tiles (256 weight rows, cluster of 2)
    int kb = 1;        // 64-column K blocks per stage (1 or 2)
    int BN = 0;        // tokens per tile (128 or 256)
    int TB = 0;        // token blocks
    int ntiles = 0;    // output tiles (128 or 256 weight rows x BN tokens)
    int S = 0;         // K splits
    int spl = 0;       // 64-column stages per split
    int nks = 0;       // stages over K
    int units = 0;     // ntiles * S
    int grid = 0;      // CTAs launched
    size_t ticket_bytes = 0;  // split-K counters at the start of the workspace
    size_t ws_bytes = 0;
};
bool plan_gemm(int M, int N, int K, int G, int sm_count, GemmPlan* plan);
// scales_b (and offs_b for asymmetric groups): the bf16 parameter layout.
// y32 (instead of y): fp32 outputs without the bias.
int launch_w4a16_gemm(const uint16_t* x, const uint8_t* packed, const float* scales,
                      const uint8_t* zeros, const float* bias, uint16_t* y, int M, int N, int K,
                      int Kp, int G, const GemmPlan& p, void* workspace, int* err,
                      cudaStream_t stream, const uint16_t* scales_b = nullptr,
                      const uint16_t* offs_b = nullptr, float* y32 = nullptr);
// Grouped (experts) prefill on the tensor cores: group e's tokens, rows
// goff[e] .. goff[e+1] - 1 of x [T, K], times its Ne x K matrix (rows
// e * Ne .. of the stacked weights), in tiles of 64 (tile <= 64) or 256
// tokens; requires K % 8 == 0 and a 16-byte aligned x.
int launch_w4a16_grouped_gemm(const uint16_t* x, const int* goff, const uint8_t* packed,
                              const float* scales, const uint8_t* zeros, const float* bias,
                              uint16_t* y, int T, int E, int Ne, int K, int Kp, int G, int tile,
                              int* err, cudaStream_t stream);
// ysum [M, N] fp32 + bias -> y bf16 (the last step of a row-parallel layer).
int launch_partial_finish(const float* ysum, const float* bias, uint16_t* y, int M, int N,
                          cudaStream_t stream);

// ---------------------------------------------------------------- others
// scales_b (and offs_b): write the bf16 parameter layout instead of fp32
// scales and uint8 zero points.
int launch_pack_rtn(const float* W, int N, int K, int G, int symmetric,
                    uint8_t* packed, float* scales, uint8_t* zeros, uint16_t* scales_b,
                    uint16_t* offs_b, cudaStream_t stream);
// inv_s: SmoothQuant column factors 1/s (nullptr: none).
int launch_act_quant(const uint16_t* x, const float* inv_s, int M, int K, int Kp, int8_t* qx,
                     float* sx, cudaStream_t stream);
// GPTQ (gptq.cu): column block width for a group size, workspace bytes,
// and the whole quantizer (Hessian .. packed codes) on one stream.
int gptq_block_cols(int G);
size_t gptq_workspace_bytes(int N, int Kp, int B);
int launch_gptq(const uint16_t* X, int T, const float* W, int N, int K, int Kp, int G,
                int symmetric, float damp, uint8_t* packed, float* scales, uint8_t* zeros,
                float* loss, void* ws, int* err, cudaStream_t st);
// SmoothQuant calibration: s, inv_s [K] from X [T, K] bf16 and W [N, K] fp32,
// then W *= s per column, in place.
int launch_smooth(const uint16_t* X, int T, float* W, int N, int K, float alpha, float* s,
                  float* inv_s, cudaStream_t stream);

}  // namespace w4
