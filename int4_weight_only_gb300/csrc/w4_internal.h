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
// Decode kernels: one CTA per SM; a unit of work is (block of 128 output
// rows, slice of the padded K).  Slices are whole 256-column stages.
constexpr int kGemvRows = 128;          // rows per unit (8 consumer warps x 16)
constexpr int kGemvStageK = 256;        // K columns per pipeline stage
constexpr int kGemvStages = 6;          // pipeline depth
constexpr int kGemvConsumerWarps = 8;
constexpr int kGemvThreads = 32 * (kGemvConsumerWarps + 1);

struct GemvPlan {
    int NB = 0;        // row blocks
    int nst = 0;       // stages over Kp
    int S = 0;         // K splits
    int spl = 0;       // stages per split
    int units = 0;     // NB * S
    int grid = 0;      // CTAs launched
    int XS = 0;        // activation row stride in shared memory (bytes)
    size_t smem = 0;   // dynamic shared memory (bytes)
    size_t ws_bytes = 0;
};

// act_bytes: bytes per activation element (2 for bf16, 1 for int8).
// Returns false if no plan fits (M too large).
bool plan_gemv(int M, int N, int Kp, int act_bytes, int sm_count, GemvPlan* plan);

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
    int nst, S, spl, units, XS;
};

int launch_w4a16_gemv(const CUtensorMap& tmW, const GemvArgs& a, const GemvPlan& p,
                      cudaStream_t stream);
int launch_w4a8_gemv(const CUtensorMap& tmW, const GemvArgs& a, const GemvPlan& p,
                     cudaStream_t stream);

// ---------------------------------------------------------------- prefill
// Tensor-core kernel for M > 16 (requires K % 8 == 0 and 16-byte aligned x).
int launch_w4a16_gemm(const uint16_t* x, const uint8_t* packed, const float* scales,
                      const uint8_t* zeros, const float* bias, uint16_t* y, int M, int N, int K,
                      int Kp, int G, int* err, int sm_count, cudaStream_t stream);

// ---------------------------------------------------------------- others
int launch_pack_rtn(const float* W, int N, int K, int G, int symmetric,
                    uint8_t* packed, float* scales, uint8_t* zeros,
                    cudaStream_t stream);
int launch_act_quant(const uint16_t* x, int M, int K, int Kp, int8_t* qx, float* sx,
                     cudaStream_t stream);

}  // namespace w4
