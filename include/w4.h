/*
 * w4.h - C ABI of libw4: the group-wise INT4 weight-only quantized linear
 * layer y = x * W_hat^T (+ b) on one NVIDIA GB300 (sm_103a).
 *
 * Definitions this library implements (page title, section):
 *
 *  [LAB5] "Lab 5: Gemma4 端到端推理优化", section "INT4 线性量化":
 *     q = clip(round(r/s + z), qmin, qmax), r_hat = s (q - z); one (s, z) per
 *     output channel and per group_size input columns.  Symmetric groups use
 *     s = max|r| / 7 and store the code q + 8 in [0, 15] (r_hat = s (code-8));
 *     asymmetric groups use s = (r_max - r_min) / 15, z = round(-r_min / s).
 *     Two codes per uint8, the earlier column in the low nibble.  K is padded
 *     up to a multiple of group_size and padded positions dequantize to 0.
 *  [LAB5-F] same page, sections "融合INT4反量化与矩阵乘" and
 *     "Prefill和Decode分流": dequantize in registers next to the matmul for
 *     small M (decode); for large M the layer is a dense GEMM.
 *  [ORIN] "Jetson Orin AGX INT4 推理优化实践：super 分支从 9 tok/s 到 24 tok/s",
 *     section "从 FP 线性层到 INT4 DP4A 的数学推导": per-row INT4 weights,
 *     per-token dynamic INT8 activations s_x = max|x| / 127,
 *     q_x = clip(round(x / s_x), -127, 127), acc_j = sum_i q^W_ji q^x_i in
 *     int32, y_j = s^W_j s_x acc_j + b_j; section "INT32 accumulator 是否安全".
 *
 * Conventions for every entry point
 *  - Matrices are row-major.  W is [N, K] (out x in); x is [M, K]; y is [M, N].
 *  - Kp = ceil(K / group_size) * group_size;  Ng = Kp / group_size.
 *  - bf16 tensors are passed as uint16_t bit patterns (IEEE bfloat16).
 *  - All data pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or synchronizes (except w4_get_device_error).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream); every
 *    call only enqueues work on it and returns.
 *  - Return value: W4_OK (0) or a negative W4_ERR_* code.  Arguments are
 *    checked on the host before anything is enqueued; a failed check leaves
 *    every output untouched.  w4_error_string() names a code.
 *  - group_size must be a positive multiple of 32 (each packed group is a
 *    whole number of 16-byte words).
 *  - Weights (packed, scales, zeros) are assumed constant while a call that
 *    reads them is in flight.
 *  - The linear entry points use programmatic dependent launch: their
 *    kernels may start, and read packed, scales, zeros and bias, while the
 *    kernel enqueued just before them on the stream is still finishing; x,
 *    the workspace and y are touched only after it has completed.  So the
 *    kernel immediately before a linear call must not write that call's
 *    weights or bias.  w4_pack_rtn ends with an empty kernel launched
 *    without this relaxation, so packing and then calling a linear layer on
 *    the same stream is safe.
 */
#ifndef W4_H_
#define W4_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W4_API __attribute__((visibility("default")))
#else
#define W4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define W4_OK                       0
#define W4_ERR_INVALID_ARG         -1  /* a size or flag is out of range      */
#define W4_ERR_NULL_PTR            -2  /* a required pointer is NULL          */
#define W4_ERR_MISALIGNED          -3  /* a buffer not aligned as the entry
                                          point states (packed, x, qx: 16 B) */
#define W4_ERR_UNSUPPORTED_GROUP   -4  /* group_size not a positive mult. of 32,
                                          or a W4A8 group size the group-wise
                                          kernel does not take               */
#define W4_ERR_K_TOO_LARGE         -5  /* W4A8: Kp * 15 * 127 >= 2^31         */
#define W4_ERR_WORKSPACE           -6  /* workspace NULL or too small         */
#define W4_ERR_CUDA                -7  /* a CUDA runtime call failed          */
#define W4_ERR_UNSUPPORTED_SHAPE   -8  /* shape outside what a kernel takes   */
#define W4_ERR_DEVICE_TIMEOUT      -9  /* a kernel's bounded wait ran out     */
#define W4_ERR_SCRATCH_LIMIT      -10  /* shape needs more split-K scratch than
                                          W4_NOALLOC_SCRATCH_BYTES            */
#define W4_ERR_GROUP_TOKENS       -11  /* device flag: a group's token offsets
                                          were invalid; its rows of y were not
                                          written                             */
#define W4_ERR_NOT_SPD            -12  /* device flag: w4_gptq met a non-positive
                                          pivot (damped Hessian not positive
                                          definite in fp32); results unreliable */

/* Size of the library's built-in split-K scratch used by
 * w4a16_linear_noalloc (4 MiB, held by every GPU that loads the library).  */
#define W4_NOALLOC_SCRATCH_BYTES (4 << 20)

/* Workspace layout of w4a16_linear / w4a8_linear: the first
 * W4_WORKSPACE_COUNTER_BYTES hold split-K arrival counters (one int32 per
 * row block or output tile), the partial sums follow.  No call writes
 * anything but counters into the prefix, so one zero-filled workspace can
 * serve calls of different shapes. */
#define W4_WORKSPACE_COUNTER_BYTES (64 << 10)

/* Largest padded K accepted by the W4A8 path: the kernels accumulate
 * code (0..15) x q_x (-127..127) products in int32, so Kp * 15 * 127 must
 * stay below 2^31 ([ORIN], "INT32 accumulator 是否安全", for the signed
 * form K * 8 * 127).                                                       */
#define W4_W4A8_MAX_KP 1127288

/* ---------------------------------------------------------------------------
 * w4_pack_rtn - round-to-nearest INT4 quantisation and packing ([LAB5]).
 *
 *  W       [N, K] fp32 input weights.
 *  packed  [N, Kp/2] uint8 out: byte j of a row holds column 2j in bits 0-3
 *          and column 2j+1 in bits 4-7; 16-byte aligned.
 *  scales  [N, Ng] fp32 out.
 *  zeros   [N, Ng] uint8 out when symmetric == 0; must be NULL when
 *          symmetric != 0 (symmetric codes are q + 8).
 *  Rounding: each division is one IEEE fp32 division rounded to nearest
 *  even, round() is round-half-to-even, pads count as zeros in the group
 *  statistics, an asymmetric range is widened to contain 0, and an all-zero
 *  group stores s = 0 (z = 0).  Codes are bit-identical to a scalar fp32
 *  evaluation of the formulas in that order.
 * ------------------------------------------------------------------------- */
W4_API int w4_pack_rtn(const float* W, int N, int K, int group_size, int symmetric,
                uint8_t* packed, float* scales, uint8_t* zeros, void* stream);

/* ---------------------------------------------------------------------------
 * w4a16_linear_noalloc - w4a16_linear for callers that cannot allocate
 * device memory: a plugin that is handed only its input and output
 * buffers, or a runtime that forbids cudaMalloc after start-up (it can
 * synchronize the device and can fail under a fixed memory budget).  The
 * pages have no counterpart; this is a library convenience.
 *
 *  Same arguments and results as w4a16_linear with M <= 16 (the decode
 *  kernel), but no workspace argument: split-K partial sums and arrival
 *  counters live in a W4_NOALLOC_SCRATCH_BYTES array inside the library.
 *  Shapes whose split needs more scratch than that return
 *  W4_ERR_SCRATCH_LIMIT before anything is enqueued; M > 16 returns
 *  W4_ERR_UNSUPPORTED_SHAPE.  Nothing is allocated: no cudaMalloc, no
 *  cudaFree.
 *  The first call on a device looks up the array's device address (with
 *  that device current); make that first call before any stream capture.
 *  Each call clears the counters on `stream` before its kernel.  All calls
 *  share the one array and it keeps the previous call's contents, so calls
 *  that overlap on the GPU (different streams or threads) race and must be
 *  serialized by the caller.
 * ------------------------------------------------------------------------- */
W4_API int w4a16_linear_noalloc(const uint16_t* x, const uint8_t* packed,
                                const float* scales, const uint8_t* zeros,
                                const float* bias, uint16_t* y, int M, int N, int K,
                                int group_size, int symmetric, void* stream);

/* ---------------------------------------------------------------------------
 * w4a16_workspace_bytes - bytes of device workspace w4a16_linear needs for
 * this shape on the CURRENT device (W4_WORKSPACE_COUNTER_BYTES of arrival
 * counters, then split-K partial sums).  May be 0.  The workspace must be
 * zero-filled once before its first use; every call leaves the counters at
 * zero again, so it can be reused by later calls of any shape on the same
 * stream without clearing.
 * ------------------------------------------------------------------------- */
W4_API size_t w4a16_workspace_bytes(int M, int N, int K, int group_size);

/* ---------------------------------------------------------------------------
 * w4a16_linear - y = x * W_hat^T (+ bias), W_hat = s (code - z) per group
 * ([LAB5]); bf16 activations and outputs, fp32 accumulation.
 *
 *  x        [M, K] bf16, 16-byte aligned.
 *  packed   [N, Kp/2] uint8 from w4_pack_rtn, 16-byte aligned.
 *  scales   [N, Ng] fp32.
 *  zeros    [N, Ng] uint8, or NULL for symmetric groups (z = 8).
 *  bias     [N] fp32 or NULL.
 *  y        [M, N] bf16 out.
 *  symmetric must agree with zeros == NULL.
 *  M <= 16 runs the decode kernel (dequantize in registers, one pass over the
 *  weights); larger M runs the tensor-core prefill kernel, which requires
 *  K % 8 == 0.  workspace: see w4a16_workspace_bytes.  Calls that share a
 *  workspace must not overlap on the GPU.
 * ------------------------------------------------------------------------- */
W4_API int w4a16_linear(const uint16_t* x, const uint8_t* packed, const float* scales,
                 const uint8_t* zeros, const float* bias, uint16_t* y,
                 int M, int N, int K, int group_size, int symmetric,
                 void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * w4a16_linear_partial / w4a16_partial_finish - one layer sharded across GPUs
 * by its input columns (row-parallel): shard s owns a group-aligned slice
 * [k0, k1) of K (k0 and k1 multiples of group_size, the last shard holding
 * the ragged end), packed by w4_pack_rtn from W[:, k0:k1] (its codes and
 * scales are exactly columns k0/2 .. k1/2 and groups k0/G .. k1/G of the
 * whole layer's), and its slice x[:, k0:k1] of the activations.  Then
 *  y = sum_s x_s W_hat_s^T + b:
 * each shard computes its fp32 partial with w4a16_linear_partial, the
 * partials are added across shards (one all-reduce, outside this library),
 * and w4a16_partial_finish adds the bias and rounds to bf16 once.  The
 * column-parallel split needs no entry point of its own: a shard's rows
 * n0 .. n1 - 1 are a w4a16_linear of the rows' slice of packed, scales,
 * zeros and bias.  The pages give the layer and its quantization, not its
 * distribution ("Lab 5: Gemma4 端到端推理优化", sections "INT4 线性量化"
 * and "Prefill和Decode分流"); the split is the usual tensor-parallel one.
 *
 *  w4a16_linear_partial: x, packed, scales, zeros, M, N, K, group_size,
 *    symmetric, workspace as for w4a16_linear (K is the slice's width);
 *    y32 [M, N] fp32 out, 4-byte aligned: sum_k x[m,k] W_hat[n,k], no bias.
 *  w4a16_partial_finish: ysum [M, N] fp32 (the sum over shards), bias [N]
 *    fp32 or NULL, y [M, N] bf16 out: y = bf16(ysum + bias).
 * ------------------------------------------------------------------------- */
W4_API int w4a16_linear_partial(const uint16_t* x, const uint8_t* packed, const float* scales,
                                const uint8_t* zeros, float* y32, int M, int N, int K,
                                int group_size, int symmetric, void* workspace,
                                size_t workspace_bytes, void* stream);
W4_API int w4a16_partial_finish(const float* ysum, const float* bias, uint16_t* y, int M, int N,
                                void* stream);

/* ---------------------------------------------------------------------------
 * w4_pack_rtn_bf16 / w4a16_linear_bf16p - the same layer with its group
 * parameters stored in bf16 (half the parameter bytes): bf16 scales, as the
 * TPU W4A16 layers load them ("Yeniden paketlenmiş QAT Gemma 4 26B-A4B, tek
 * bir TPU v6e'de FP8 işlemenin 1.9 katı verimle sunuluyor", section 26B'deki
 * boşluk), and for asymmetric groups the additive offset (8 - z) s of
 * codes read as (code - 8) ("Lab 5: Gemma4 端到端推理优化", section
 * 融合INT4反量化与矩阵乘) instead of the zero point:
 *  w_hat = s_b (code - 8) + o_b,  s_b = bf16(s),  o_b = bf16(fp32((8 - z) s))
 * (round to nearest even).  The codes are exactly w4_pack_rtn's.
 *
 *  w4_pack_rtn_bf16: W, N, K, group_size, symmetric, packed as for
 *    w4_pack_rtn; scales_b [N, Ng] bf16 out; offsets_b [N, Ng] bf16 out when
 *    symmetric == 0, else NULL.
 *  w4a16_linear_bf16p: as w4a16_linear (same shapes, plans, workspace);
 *    scales_b and offsets_b (NULL: symmetric) 16-byte aligned.
 * ------------------------------------------------------------------------- */
W4_API int w4_pack_rtn_bf16(const float* W, int N, int K, int group_size, int symmetric,
                            uint8_t* packed, uint16_t* scales_b, uint16_t* offsets_b,
                            void* stream);
W4_API int w4a16_linear_bf16p(const uint16_t* x, const uint8_t* packed, const uint16_t* scales_b,
                              const uint16_t* offsets_b, const float* bias, uint16_t* y, int M,
                              int N, int K, int group_size, void* workspace,
                              size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * w4a16_linear_swiglu - the gate and up projections of a SwiGLU feed-forward
 * layer in one pass, y = SiLU(x W_gate^T + b_gate) (*) (x W_up^T + b_up),
 * SiLU(v) = v * sigmoid(v).  "Lab 5: Gemma4 端到端推理优化", section 基础
 * (FFN(x) = W_down [SiLU(W_gate x) (*) (W_up x)]); fusing SwiGLU into the
 * linear is the "kernel fusion" direction of "Jetson Orin AGX INT4
 * 推理优化实践", section 后续还能继续优化什么.
 *
 *  The weights are the 2F x K matrix whose 16-row tiles hold 8 gate rows
 *  followed by the same 8 up rows (gate row f is row 16 (f/8) + f%8, up row f
 *  is 8 rows below it), quantized and packed by w4_pack_rtn like any other;
 *  bias (optional) is ordered the same way, [2F] fp32.  F % 8 == 0.
 *  x [M, K] bf16, y [M, F] bf16 out.  M <= 16 (the decode kernel; larger M
 *  returns W4_ERR_UNSUPPORTED_SHAPE).  workspace: w4a16_workspace_bytes(M,
 *  2F, K, group_size) bytes, as for w4a16_linear.
 * ------------------------------------------------------------------------- */
W4_API int w4a16_linear_swiglu(const uint16_t* x, const uint8_t* packed, const float* scales,
                               const uint8_t* zeros, const float* bias, uint16_t* y, int M,
                               int F, int K, int group_size, int symmetric, void* workspace,
                               size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * w4a16_linear_swiglu_q8 - w4a16_linear_swiglu that also emits the INT8
 * activations of the W4A8 layer that follows it, in the same launch: the
 * per-token dynamic quantization folded into the op before the integer
 * GEMV ("Jetson Orin AGX INT4 推理优化实践", section 后续还能继续优化什么,
 * item 2; the rule of [ORIN], as w4a8_quantize_act applies it to y):
 *  y        as w4a16_linear_swiglu, [M, F] bf16 out, 16-byte aligned;
 *  qx       [M, Fp] int8 out, Fp = ceil(F / q_group_size) * q_group_size,
 *           16-byte aligned, columns F .. Fp-1 zero;
 *  sx       [M] fp32 out;
 *  q_group_size  the group size of the W4A8 layer that reads qx (a positive
 *           multiple of 32; its padded K is Fp).
 * qx and sx equal w4a8_quantize_act(y, q_group_size) bit for bit.  Each
 * CTA folds the max |y| per token of the outputs it wrote into the
 * workspace; after a grid-wide barrier (the kernel is launched
 * cooperatively when the device allows it) every CTA quantizes a share of
 * y, else the last CTA to finish quantizes all of it.  The workspace is
 * therefore required even when the plan does not split K: at least
 * max(w4a16_workspace_bytes(M, 2F, K, group_size), W4_WORKSPACE_COUNTER_BYTES)
 * bytes, zero-filled once (its counters are left at zero).  M <= 16.
 * ------------------------------------------------------------------------- */
W4_API int w4a16_linear_swiglu_q8(const uint16_t* x, const uint8_t* packed,
                                  const float* scales, const uint8_t* zeros,
                                  const float* bias, uint16_t* y, int8_t* qx, float* sx,
                                  int M, int F, int K, int group_size, int symmetric,
                                  int q_group_size, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* ---------------------------------------------------------------------------
 * w4a16_grouped_linear - grouped W4A16 linear over E groups (mixture-of-
 * experts layers), decode sizes: tokens sorted by group, each group's tokens
 * multiplied by that group's own quantized matrix in one launch:
 *  y[t, n] = sum_k x[t, k] * W_hat_e[n, k] (+ bias[e, n])
 *  for goff[e] <= t < goff[e+1].
 * The grouped matmul of "Yeniden paketlenmiş QAT Gemma 4 26B-A4B, tek bir
 * TPU v6e'de FP8 işlemenin 1.9 katı verimle sunuluyor" (expert layers: 128
 * experts, 8 active per token, int4 with 32-wide groups, each weight chunk
 * dequantized on chip before the multiply), sections "26B'deki boşluk" and
 * "vLLM'in TPU backend'inde değişen ne oldu"; the per-group formula is
 * w4a16_linear's.
 *
 *  x         [T, K] bf16, rows sorted by group, 16-byte aligned.
 *  goff      [E+1] int32 on the device, non-decreasing, goff[0] = 0,
 *            goff[E] = T (group e's tokens are rows goff[e] .. goff[e+1]-1).
 *            Read on the device after the previous kernel on the stream has
 *            finished, so a router kernel may write it just before.
 *  packed    [E, N, Kp/2] uint8 (w4_pack_rtn of the stacked [E*N, K] weights);
 *  scales    [E, N, Ng] fp32;  zeros [E, N, Ng] uint8 or NULL (symmetric);
 *  bias      [E, N] fp32 or NULL.
 *  y         [T, N] bf16 out.
 *  tile_tokens  tokens per pass.  1..16: the decode kernel (token tiles 8
 *            or 16 wide); a group with more tokens is taken in
 *            ceil(count / tile_tokens) passes, each reading its weights; the
 *            best tile is the largest count of a group when that is <= 16.
 *            17..256: the tensor-core (tcgen05) kernel for groups of many
 *            tokens (prefill), in tiles of 64 tokens (tile_tokens <= 64) or
 *            256, each tile dequantizing its group's weights on chip once;
 *            requires K % 8 == 0 and supports up to a few hundred groups
 *            (W4_ERR_UNSUPPORTED_SHAPE beyond).
 *  A group whose offsets lie outside [0, T] or decrease is skipped (its rows
 *  of y are left as they were) and sets W4_ERR_GROUP_TOKENS in the device
 *  flag that w4_get_device_error returns.  Groups without tokens cost
 *  nothing: the units of work are ((group, token tile), row block), listed
 *  on the device.  E <= 32767, E * N < 2^31, T / tile_tokens < 65536 (decode
 *  tiles).  No workspace (grouped plans do not split K).
 * ------------------------------------------------------------------------- */
W4_API int w4a16_grouped_linear(const uint16_t* x, const int32_t* goff, const uint8_t* packed,
                                const float* scales, const uint8_t* zeros, const float* bias,
                                uint16_t* y, int T, int E, int N, int K, int group_size,
                                int symmetric, int tile_tokens, void* stream);

/* ---------------------------------------------------------------------------
 * w4_gptq - GPTQ quantization of one linear layer on the GPU, in FP32
 * ("Lab 5: Gemma4 端到端推理优化", section 从 RTN 到 GPTQ):
 *  H = (2/T) X^T X; a dead column (H_jj = 0, also every padded column
 *  K..Kp-1) gets W[:, j] = 0 and H_jj = 1; H += damp * mean(diag H) I;
 *  H^-1 = U^T U (U upper); then for each column i in order: the group's
 *  parameters, when i is its first column, from its current weights by the
 *  rule of w4_pack_rtn; q_i by that rule; e_i = (w_i - q_i) / U_ii;
 *  W[:, i:] -= e_i U[i, i:];  loss[n] = 1/2 sum_i (w_i - q_i)^2 / U_ii^2.
 *
 *  X        [T, K] bf16 calibration activations, T >= 1.
 *  W        [N, K] fp32 weights (read only).
 *  group_size, symmetric: as for w4_pack_rtn; damp >= 0 (0.01 typical).
 *  packed [N, Kp/2], scales [N, Ng], zeros [N, Ng] (asymmetric, else NULL):
 *           out, the w4_pack_rtn layout.
 *  loss     [N] fp32 out (L_pred per row).
 *  workspace: w4_gptq_workspace_bytes(N, K, group_size) bytes, 256-byte
 *           aligned; its contents need no initialisation.
 *  A non-positive Cholesky pivot sets W4_ERR_NOT_SPD in the device flag.
 * ------------------------------------------------------------------------- */
W4_API size_t w4_gptq_workspace_bytes(int N, int K, int group_size);
W4_API int w4_gptq(const uint16_t* X, int T, const float* W, int N, int K, int group_size,
                   int symmetric, float damp, uint8_t* packed, float* scales, uint8_t* zeros,
                   float* loss, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * w4a8_quantize_act - per-token dynamic INT8 activations ([ORIN]):
 *  s_x[m] = fp32(max_k |x[m,k]| / 127),
 *  qx[m,k] = clip(round(fp32(x[m,k] / s_x[m])), -127, 127) for k < K, 0 for
 *  K <= k < Kp; an all-zero token gets s_x = 0 and qx = 0.
 *
 *  x   [M, K] bf16;  qx [M, Kp] int8 out (16-byte aligned);  sx [M] fp32 out.
 * ------------------------------------------------------------------------- */
W4_API int w4a8_quantize_act(const uint16_t* x, int M, int K, int group_size,
                      int8_t* qx, float* sx, void* stream);

/* ---------------------------------------------------------------------------
 * w4a8_quantize_act_smooth - w4a8_quantize_act on SmoothQuant-smoothed
 * activations ("【infra之路】12-投机解码、量化与推理引擎对比", section 2.4:
 * Y = (X diag(s)^-1)(diag(s) W)): x'[m,k] = fp32(x[m,k] * inv_s[k]) (one
 * rounding), then s_x and qx from x' by the rule above.  The weights must
 * carry the factors (w4_smooth) before they are packed.
 *
 *  inv_s  [K] fp32, 16-byte aligned (1/s from w4_smooth).
 *  Other arguments and outputs as for w4a8_quantize_act.
 * ------------------------------------------------------------------------- */
W4_API int w4a8_quantize_act_smooth(const uint16_t* x, const float* inv_s, int M, int K,
                                    int group_size, int8_t* qx, float* sx, void* stream);

/* ---------------------------------------------------------------------------
 * w4_smooth - SmoothQuant calibration of one linear layer (same section; the
 * factor range and per-layer tuning of alpha: "LLM 模型壓縮與推理加速實踐-
 * 陳磊.pdf", W8A8 slides):
 *  s[j]     = max_t |X[t,j]|^alpha / max_n |W[n,j]|^(1 - alpha)  (fp32 powf;
 *             1 where either maximum is 0),  inv_s[j] = fp32(1 / s[j]),
 *  W[n,j]  *= s[j]  (in place; pack W afterwards with w4_pack_rtn).
 *
 *  X      [T, K] bf16 calibration activations (T >= 0; T = 0 gives s = 1).
 *  W      [N, K] fp32, device, modified.
 *  alpha  in [0, 1] (0.5 typical).
 *  s, inv_s  [K] fp32 out (device).
 *  Ends with an ordinary (not programmatic) launch, like w4_pack_rtn.
 * ------------------------------------------------------------------------- */
W4_API int w4_smooth(const uint16_t* X, int T, float* W, int N, int K, float alpha, float* s,
                     float* inv_s, void* stream);

/* ---------------------------------------------------------------------------
 * w4a8_workspace_bytes - as w4a16_workspace_bytes, for w4a8_linear.
 * ------------------------------------------------------------------------- */
W4_API size_t w4a8_workspace_bytes(int M, int N, int K, int group_size);

/* ---------------------------------------------------------------------------
 * w4_decode_plan - the launch plan the library picks for a decode call
 * (M <= 16) of one layer, computed on the host alone: no device is touched,
 * so it answers for any SM count, with or without a GPU.  The pages have no
 * counterpart; it exposes the library's own planner for inspection and
 * tests.
 *
 *  kind      0: w4a16_linear (and the calls that share its plans:
 *            _partial, _bf16p, _noalloc); 1: w4a8_linear (per-row or
 *            group-wise scales).
 *  M, N, K, group_size  as for those calls; 1 <= M <= 16.
 *  sm_count  SMs of the device the plan is for (152 on a GB300).
 *  out       host array of W4_DECODE_PLAN_FIELDS int64, written on success:
 *    [0] rows of a unit (16, 32, 64 or 128)   [1] K splits S
 *    [2] stages per split                      [3] stages over the padded K
 *    [4] K columns per stage (32768 / rows: 16 KB of packed codes)
 *    [5] units (row blocks x S)                [6] CTAs launched
 *    [7] CTAs per SM the plan is sized for     [8] dynamic shared memory per
 *        CTA (bytes)                            [9] workspace bytes (0
 *        without a K split; else W4_WORKSPACE_COUNTER_BYTES + S*M*N*4)
 *    [10] 1: the fp16 inner loop (1-2 tokens), 0: bf16 (W4A16) or int8
 *    [11] 1: the K splits hand off inside a thread-block cluster, 0: the
 *         global last-arriver hand-off (or no split)
 *  The tuning variables W4_GEMV_ROWS, W4_GEMV_SPLIT, W4_GEMV_CPS,
 *  W4_GEMV_F16 and W4_GEMV_CSPLIT apply as they do to the calls.
 *  Returns W4_ERR_NULL_PTR, W4_ERR_INVALID_ARG (kind, M, N, K or sm_count
 *  out of range), W4_ERR_UNSUPPORTED_GROUP, W4_ERR_K_TOO_LARGE (kind 1) or
 *  W4_ERR_UNSUPPORTED_SHAPE (no plan fits) as the calls would.
 * ------------------------------------------------------------------------- */
#define W4_DECODE_PLAN_FIELDS 12
W4_API int w4_decode_plan(int kind, int M, int N, int K, int group_size, int sm_count,
                          long long* out);

/* ---------------------------------------------------------------------------
 * w4a8_linear - INT4 x INT8 integer linear layer ([ORIN]):
 *  acc[m,n] = sum_{k < Kp} (code[n,k] - 8) * qx[m,k]   (exact, int32)
 *  y[m,n]   = s_W[n] * s_x[m] * acc[m,n] + bias[n]      (fp32, stored bf16)
 *  With group_size < Kp (group-wise weight scales, the per-group use of the
 *  INT8 rule of "【infra之路】12-投机解码、量化与推理引擎对比", section 2.2):
 *  acc_g[m,n] = sum over group g's columns of (code - 8) * qx  (int32)
 *  y[m,n]     = s_x[m] * sum_g s_W[n,g] * acc_g[m,n] + bias[n]  (fp32 sums)
 *
 *  qx, sx     from w4a8_quantize_act (same K and group_size).
 *  packed     [N, Kp/2] uint8 symmetric codes from w4_pack_rtn, 16-byte
 *             aligned; group_size == Kp (one scale per row) or, group-wise,
 *             32, 64, 128 or a multiple of 256 (else W4_ERR_UNSUPPORTED_GROUP).
 *  w_scales   [N, Ng] fp32 (Ng = Kp / group_size; [N] per row).
 *  bias       [N] fp32 or NULL.
 *  y          [M, N] bf16 out.
 *  acc_out    [M, N] int32 out, or NULL; per-row only (group-wise: must be
 *             NULL, else W4_ERR_INVALID_ARG).
 *  Requires M <= 16 and Kp <= W4_W4A8_MAX_KP.
 * ------------------------------------------------------------------------- */
W4_API int w4a8_linear(const int8_t* qx, const float* sx, const uint8_t* packed,
                const float* w_scales, const float* bias, uint16_t* y,
                int32_t* acc_out, int M, int N, int K, int group_size,
                void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * w4_get_device_error - synchronizes `stream`, then returns and clears the
 * library's device-side error flag on the current device: W4_OK, or
 * W4_ERR_DEVICE_TIMEOUT when a kernel gave up on a bounded wait (its outputs
 * are then unspecified).  Returns W4_ERR_CUDA if the synchronization fails.
 * ------------------------------------------------------------------------- */
W4_API int w4_get_device_error(void* stream);

/* ---------------------------------------------------------------------------
 * w4_set_wait_limit - how long a bounded wait inside the library's kernels
 * (a stage of a copy pipeline, a device-side list) may take before the
 * kernel gives up: it then raises W4_ERR_DEVICE_TIMEOUT in the device flag,
 * every thread of the CTA leaves its loops, the copies it already issued are
 * allowed to land (these drains always use the default limit), and the
 * call's outputs are unspecified.  A wait whose data does arrive can outlast
 * the limit, since the hardware suspends a waiting thread until its barrier
 * completes or its own time-out; with w4_set_fault_injection a wait that can
 * never complete runs out, which is how this path is tested without a fault.
 *
 *  cycles  SM clock cycles; <= 0 restores the default (2e9, about one second
 *          on a GB300).  Applies to the current device, to kernels that start
 *          after the value is written: the write is enqueued on `stream`.
 * ------------------------------------------------------------------------- */
W4_API int w4_set_wait_limit(long long cycles, void* stream);

/* ---------------------------------------------------------------------------
 * w4_set_fault_injection - a switch for failure tests: it makes one wait of
 * the grouped decode kernel (w4a16_grouped_linear) impossible to complete,
 * so that the bounded-wait path above runs without any fault.  The pages
 * have no counterpart; it exists to test the library.
 *
 *  mode  0: off (the default).  1: the kernel's consumers never publish the
 *        list of groups, so its copy producer waits until the limit and
 *        issues nothing.  2: the consumers never free a slot of the copy
 *        ring, so the producer waits until the limit with copies in flight,
 *        which it lets land before its CTA exits.  Either way the call
 *        returns, W4_ERR_DEVICE_TIMEOUT is raised, and its outputs are
 *        unspecified.  Other entry points ignore the switch.
 *  Enqueued on `stream`, for kernels that start after it; applies to the
 *  current device.  Returns W4_ERR_INVALID_ARG for other modes.
 * ------------------------------------------------------------------------- */
W4_API int w4_set_fault_injection(int mode, void* stream);

/* w4_error_string - static description of a W4_* code (never NULL). */
W4_API const char* w4_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* W4_H_ */
