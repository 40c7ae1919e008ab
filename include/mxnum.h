/*
 * mxnum.h -- C ABI of libmxnum.so: block-scaled microscaling numerics on GB300 (sm_103a).
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless stated otherwise; the caller owns every buffer and the
 *     stream.  The library allocates nothing.
 *   - Calls validate their arguments on the host and then enqueue work asynchronously on `stream`.
 *     A non-MX_OK return means nothing was enqueued (MX_ERR_CUDA: a launch failed; the CUDA error
 *     is left for the caller to query).  Outputs are valid once the stream reaches the call.
 *   - BF16 tensors are row-major 16-bit words.  Codes are row-major bytes: MXFP8 one E4M3 byte per
 *     element; NVFP4 two E2M1 codes per byte, the even-indexed element in the low nibble.
 *   - Every quantized operand keeps its blocks contiguous along the consuming GEMM's K dimension,
 *     so column-wise copies are stored transposed.
 *   - Scale bytes (E8M0 for MXFP8, E4M3 for NVFP4) are written in the block-scaled GEMM's layout:
 *     512-byte tiles of 128 rows x 4 scale columns in row-major tile order; inside a tile the scale
 *     of (row r, scale column c) sits at (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4).  Rows are
 *     padded to a multiple of 128 and scale columns to a multiple of 4; the quantizers write zeros
 *     into the padding.  mx_scale_bytes() gives the size.
 *   - Pointers to codes, scales, BF16 tensors and workspaces must be 16-byte aligned
 *     (MX_ERR_ALIGNMENT otherwise); leading dimensions are in elements and must keep rows 16-byte
 *     aligned.
 *
 * Sources (web pages): "Miles Blackwell RL ... MXFP8 e NVFP4 Nativos" (remio.ai); "NVFP4 RL
 * training" (socker-news); "End-to-End MXFP8 Reinforcement Learning on Blackwell"
 * (thelatestinai.com 2610.34915); "Train models faster with JAX and MaxText using NVFP4 on NVIDIA
 * Blackwell" (developer.nvidia.cn).  Each declaration names the passage that defines it.
 */
#ifndef MXNUM_H
#define MXNUM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MX_OK = 0,
    MX_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad enum value              */
    MX_ERR_ALIGNMENT = 2,     /* a pointer or leading dimension breaks 16-byte alignment       */
    MX_ERR_UNSUPPORTED = 3,   /* a size is not a multiple of the block or tile it needs        */
    MX_ERR_CUDA = 4,          /* a CUDA launch or runtime call failed                          */
    MX_ERR_TIMEOUT = 5        /* a device-side bounded wait gave up (see mx_check_device_status) */
} mx_status;

typedef enum { MX_FMT_MXFP8 = 0, MX_FMT_NVFP4 = 1 } mx_format;

/* Largest number of expert groups the grouped entry points accept. */
#define MX_MAX_GROUPS 1024
typedef enum { MX_ROUND_RNE = 0, MX_ROUND_SR = 1 } mx_round;
/* Scope of an FP32 second-level scale / GEMM epilogue factor. */
typedef enum { MX_SCOPE_NONE = 0, MX_SCOPE_TENSOR = 1, MX_SCOPE_ROW = 2, MX_SCOPE_GROUP = 3 } mx_scope;

/* Human-readable name of a status code (static storage). */
const char* mx_status_string(mx_status s);

/* Bytes of a scale tensor in the GEMM layout for `rows` rows whose K extent is `k` elements with
 * one scale per `block` elements (32 for MXFP8, 16 for NVFP4): ceil(rows/128) * ceil(k/block/4) * 512. */
int64_t mx_scale_bytes(int64_t rows, int64_t k, int block);

/* MXFP8 quantize, row-wise and/or column-wise in one pass over x.
 * Source: Miles page -- MXFP8 = blocks of 32 E4M3 values sharing one E8M0 scale; TransformerEngine
 * makes row-wise and column-wise copies from the high-precision input, never re-quantizing FP8
 * (section "Um Quantizador Compartilhado"); E2E page Table 10 F6 (E8M0 keeps only the exponent).
 * Per block: e = clamp(floor(log2 amax) - 8, -127, 127) (amax = 0 -> -127), scale byte = e + 127,
 * code = E4M3 round-to-nearest-even, saturating, of x * 2^-e.
 *   x      [rows, ldx] BF16 (ldx >= cols)
 *   q_row  [rows, cols] E4M3, s_row mx_scale_bytes(rows, cols, 32)   -- blocks along cols (NULL: skip)
 *   q_col  [cols, rows] E4M3, s_col mx_scale_bytes(cols, rows, 32)   -- blocks along rows, stored
 *          transposed (NULL: skip).  At least one of the two outputs must be given.
 * Requires cols % 32 == 0 for row-wise, rows % 32 == 0 for column-wise, cols % 8 == 0. */
mx_status mx_quantize_mxfp8(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                            uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                            cudaStream_t stream);

/* Several tensors through mx_quantize_mxfp8 in one launch (for instance the input, weight and output
 * gradient of a linear layer, which the training step quantizes back to back): the tiles of all the
 * tensors share one persistent grid, so the launch ramps up and drains once.  Codes and scales are
 * exactly those of one mx_quantize_mxfp8 call per tensor.
 *   tensors  HOST array of `count` descriptors (1 <= count <= MX_MXFP8_MAX_BATCH), each with the
 *            arguments and requirements of mx_quantize_mxfp8; every tensor must request the same
 *            outputs (all row-wise, all column-wise or all both), else MX_ERR_INVALID_ARG.
 * The descriptors are read before the call returns; the device buffers they name must stay valid
 * until the work on `stream` completes. */
#define MX_MXFP8_MAX_BATCH 4
typedef struct {
    const void* x;
    int64_t rows, cols, ldx;
    uint8_t* q_row;
    uint8_t* s_row;
    uint8_t* q_col;
    uint8_t* s_col;
} mx_mxfp8_tensor;
mx_status mx_quantize_mxfp8_batched(const mx_mxfp8_tensor* tensors, int count, cudaStream_t stream);

/* NVFP4 1x16 quantize with a per-token FP32 second-level scale, fused in one kernel.
 * Source: Miles page -- NVFP4 = E2M1 values, one E4M3 scale per 16, a second FP32 scale computed
 * separately for each token, online, fused into the activation quantizer that emits packed FP4,
 * block scales and token scales together; NVFP4 RL page, "Baseline recipe details".
 * Per token t: S_t = amax_t / 2688; per 16-block: bs = E4M3(amax_b / 6 / S_t) (S_t = 0 -> 0);
 * r = 1 / (bs * S_t) (0 if bs * S_t = 0, clamped to FLT_MAX); code = E2M1 RNE saturating of x * r;
 * every operation FP32 round-to-nearest in that order.
 *   x [T, ldx] BF16;  q [T, H/2];  s mx_scale_bytes(T, H, 16);  s_tok [T] FP32.
 * Requires H % 16 == 0. */
mx_status mx_nvfp4_quantize_per_token(const void* x, int64_t T, int64_t H, int64_t ldx,
                                      uint8_t* q, uint8_t* s, float* s_tok, cudaStream_t stream);

/* Grouped scale layout for expert-sorted rows (the A operand of mx_grouped_scaled_gemm): the
 * scales of group g's rows [off[g], off[g+1]) start on a 128-row tile of the GEMM layout, at padded
 * row P_g = sum over j < g of ceil(m_j / 128) * 128; row r of group g sits at padded row
 * P_g + (r - off[g]).  The rows between groups are zero.  Codes stay in plain row order.
 * Source: Miles page -- NVFP4 on the routed experts; E2E page Table 6 and Table 10 F3 (a separate
 * scale rearrangement costs time and can go stale, so the quantizer writes the GEMM's layout).
 * mx_grouped_scale_bytes(rows, G, k, block) = mx_scale_bytes(rows + 127 * G, k, block) bounds it. */
int64_t mx_grouped_scale_bytes(int64_t rows, int64_t G, int64_t k, int block);

/* mx_nvfp4_quantize_per_token for expert-sorted rows: identical codes and token scales, block
 * scales in the grouped scale layout.  group_offsets: DEVICE int64 [G + 1] (as for
 * mx_grouped_scaled_gemm); s: mx_grouped_scale_bytes(T, G, H, 16) bytes.  1 <= G <= MX_MAX_GROUPS. */
mx_status mx_nvfp4_quantize_per_token_grouped(const void* x, int64_t T, int64_t H, int64_t ldx, int64_t G,
                                              const int64_t* group_offsets, uint8_t* q, uint8_t* s,
                                              float* s_tok, cudaStream_t stream);

/* mx_quantize_mxfp8 row-wise for expert-sorted rows: identical codes, scales in the grouped scale
 * layout.  s_row: mx_grouped_scale_bytes(rows, G, cols, 32) bytes.  1 <= G <= MX_MAX_GROUPS. */
mx_status mx_quantize_mxfp8_grouped(const void* x, int64_t rows, int64_t cols, int64_t ldx, int64_t G,
                                    const int64_t* group_offsets, uint8_t* q_row, uint8_t* s_row,
                                    cudaStream_t stream);

/* NVFP4 16x16 2D weight quantize, both orientations, for G stacked matrices.
 * Source: MaxText page, "NVFP4 pretraining recipe" -- one FP8 scale per 16x16 weight block so that
 * FPROP and its transpose DGRAD see identical values, under a per-tensor FP32 scale; Miles page --
 * SwiGLU gate and up are quantized together (stack them into one matrix to share the scale).
 * Per matrix g: S_w = amax / 2688; per 16x16 tile: bs as above with the tile amax; codes as above.
 *   w      [G, O, H] BF16 (contiguous)
 *   q_row  [G, O, H/2];  s_row G * mx_scale_bytes(O, H, 16)   (tile scale on each of its 16 rows)
 *   q_col  [G, H, O/2];  s_col G * mx_scale_bytes(H, O, 16)   (the same codes, transposed)
 *   s_w    [G] FP32
 *   workspace: mx_workspace_bytes(MX_WS_WEIGHT_2D, G, 0) bytes, 16-byte aligned, caller-owned.
 * Requires O % 16 == 0 and H % 16 == 0; G <= 65535 and O <= 65535 * 64 (grid limits), else
 * MX_ERR_UNSUPPORTED.  The same limits hold for every 2D weight entry point below. */
mx_status mx_nvfp4_quantize_weight_2d(const void* w, int64_t G, int64_t O, int64_t H,
                                      uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                      float* s_w, void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream);

/* Four-over-Six variants of the two NVFP4 quantizers above.
 * Source: NVIDIA RL blog, "Four-Over-Six (4/6)" for weights and activations -- instead of always mapping
 * a block's maximum to the E2M1 maximum 6, map it to 4 or to 6, whichever errs less (the largest
 * error drops from 1/6 to 1/8 of the range); applied to activations in pretraining and also to
 * weights in RL.  Readings: per block (1x16 per token, 16x16 for weights) both candidates
 *   bs_m = E4M3(fp32(fp32(amax_b / m) / S)), m in {6, 4}, codes as above with bs_m,
 * are formed, and the one with the smaller largest |fp32(fp32(value(q) * value(bs_m)) * S) - x| is kept
 * (a tie keeps 6).  The FP32 second-level scales are unchanged (amax / 2688), so the codes and scales
 * are consumed exactly like those of the standard quantizers (GEMMs, dequantize).
 * Same arguments, sizes, alignment and error rules as mx_nvfp4_quantize_per_token and
 * mx_nvfp4_quantize_weight_2d. */
mx_status mx_nvfp4_quantize_per_token_46(const void* x, int64_t T, int64_t H, int64_t ldx, uint8_t* q, uint8_t* s,
                                         float* s_tok, cudaStream_t stream);
mx_status mx_nvfp4_quantize_weight_2d_46(const void* w, int64_t G, int64_t O, int64_t H,
                                         uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                         float* s_w, void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream);

/* Allocation-free variant of mx_nvfp4_quantize_weight_2d (the pages have no counterpart: it exists
 * for callers that cannot allocate device memory, e.g. a plugin inside a host framework that owns
 * all device memory, or a loop that must not call cudaMalloc because it synchronizes the device).
 * Same arguments, results and rules as mx_nvfp4_quantize_weight_2d, without the workspace: the
 * per-matrix scratch is a fixed array of MX_NOALLOC_MAX_MATRICES 32-bit words (16 KiB) inside the
 * library, which every GPU that loads the library keeps until the process exits.
 *   - G > MX_NOALLOC_MAX_MATRICES is rejected with MX_ERR_UNSUPPORTED (nothing is enqueued).
 *   - The first call on each device looks up the scratch address on the host (once per device);
 *     make that first call before any stream capture.  The address is cached for the life of the
 *     process: after cudaDeviceReset (or anything else that destroys the device's primary context)
 *     the cached address is stale, so do not call this entry point on that device again.
 *   - The call itself allocates nothing.  It clears the scratch it uses on `stream` before use.
 *   - All calls share the one array: calls that may overlap on the GPU (different streams, or
 *     different host threads, without ordering between them) race and must be serialized by the
 *     caller. */
#define MX_NOALLOC_MAX_MATRICES 4096
mx_status mx_nvfp4_quantize_weight_2d_noalloc(const void* w, int64_t G, int64_t O, int64_t H,
                                              uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                              float* s_w, cudaStream_t stream);

/* Blockwise FP8 quantize of activations or gradients: [1, 128] tiles, one scale per tile.
 * Source: NVIDIA NeMo RL FP8 page, "FP8 nas camadas lineares" -- E4M3 values; input activations and
 * output gradients in [1, 128] tiles with an FP32 scale each (the DeepSeek-V3 recipe); "Opções
 * avançadas" -- power-of-two scales instead of FP32.  Per tile, amax = max |x|:
 *   pow2 = 0:  s = fp32(amax / 448), code = E4M3 (RNE, saturating) of fp32(x / s); amax = 0 gives s = 0
 *              and signed-zero codes.
 *   pow2 = 1:  k = the smallest integer with 448 * 2^k >= amax, clamped to [-127, 127] (amax = 0 gives
 *              -127); s = 2^k; code = E4M3 of x * 2^-k (exact scaling, one rounding).
 * Row-wise tiles run along cols; column-wise tiles run along rows (the copy a GEMM contracting over
 * rows consumes, e.g. the weight gradient), stored transposed.  Both copies come from one read of x.
 *   x       [rows, ldx] BF16 (ldx >= cols)
 *   q_row   [rows, cols] E4M3, s_row [rows, cols/128] FP32            (NULL q_row: skip row-wise)
 *   sf_row  pow2 only (else NULL): mx_scale_bytes(rows, cols, 32) bytes, E8M0 byte k + 127 of each tile
 *           repeated over its four 32-element sub-blocks in the MXFP8 GEMM scale layout, so q_row and
 *           sf_row are an MXFP8 GEMM operand decoding to the same values (NULL: skip)
 *   q_col   [cols, rows] E4M3, s_col [cols, rows/128] FP32            (NULL q_col: skip column-wise)
 *   sf_col  pow2 only: mx_scale_bytes(cols, rows, 32) bytes, as sf_row for q_col (NULL: skip)
 * Requires cols % 128 == 0 for row-wise, rows % 128 == 0 for column-wise, cols % 16 == 0, ldx % 8 == 0,
 * rows * cols / 128 < 2^31; pointers 16-byte aligned.  The rows/cols of the GEMM layout padding are not written. */
mx_status mx_fp8_blockwise_quantize_1x128(const void* x, int64_t rows, int64_t cols, int64_t ldx, int pow2,
                                          uint8_t* q_row, float* s_row, uint8_t* sf_row,
                                          uint8_t* q_col, float* s_col, uint8_t* sf_col, cudaStream_t stream);

/* Blockwise FP8 quantize of weights: [128, 128] blocks, one scale per block, codes in both
 * orientations (the forward GEMM reads [O, H] with blocks along H, the data-gradient GEMM reads
 * [H, O] with blocks along O; a square block has one scale for both).
 * Source: NVIDIA NeMo RL FP8 page, "FP8 nas camadas lineares" -- weights in [128, 128] blocks with an
 * FP32 scale each; "Opções avançadas" -- power-of-two scales.  Scale and code rules as in
 * mx_fp8_blockwise_quantize_1x128 with the block's amax; the last block row / column may be partial.
 *   w      [G, O, H] BF16, G stacked matrices (experts)
 *   q_row  [G, O, H] E4M3;  q_col [G, H, O] E4M3 (the same codes transposed)
 *   s      [G, ceil(O/128), ceil(H/128)] FP32
 *   sf_row pow2 only (else NULL): G x mx_scale_bytes(O, H, 32) bytes, MXFP8 GEMM layout for q_row (NULL: skip)
 *   sf_col pow2 only: G x mx_scale_bytes(H, O, 32) bytes, for q_col (NULL: skip)
 * Requires O % 16 == 0 and H % 16 == 0 (O % 128 == 0 and H % 128 == 0 when sf_row / sf_col is given);
 * pointers 16-byte aligned. */
mx_status mx_fp8_blockwise_quantize_128x128(const void* w, int64_t G, int64_t O, int64_t H, int pow2,
                                            uint8_t* q_row, uint8_t* q_col, float* s,
                                            uint8_t* sf_row, uint8_t* sf_col, cudaStream_t stream);

/* 16-point random Hadamard transform along the token dimension.
 * Source: MaxText page, "NVFP4 pretraining recipe" -- a random Hadamard transform on the WGRAD
 * inputs only, to Gaussianize outliers before 4-bit quantization.
 * For every column n and aligned 16-token chunk: v = d * x (signs d_j = bit j of word 0 of
 * Philox4x32-10(key = seed, ctr = (0,0,1,0)), set bit = -1); Walsh-Hadamard butterflies with
 * strides 1, 2, 4, 8 in FP32; y = BF16 RNE of v / 4.  Use the same seed for both WGRAD operands.
 *   x, y [T, N] BF16 (may not alias).  Requires T % 16 == 0 and N % 8 == 0. */
mx_status mx_rht16(const void* x, int64_t T, int64_t N, uint64_t seed, void* y, cudaStream_t stream);

/* NVFP4 1x16 quantize with a per-tensor FP32 second-level scale; column-wise (blocks of 16 along
 * the token dim T, output transposed) or row-wise; optional RHT first; RNE or stochastic rounding.
 * Source: MaxText page, "NVFP4 pretraining recipe" -- 1x16 scaling for activations and gradients,
 * per-tensor FP32 scale, RHT on WGRAD inputs, SR on gradients (RNE on weights and activations).
 * Pass 1: A = amax of the (transformed, BF16-rounded) tensor; S = A / 2688.  Pass 2: per block as in
 * mx_nvfp4_quantize_per_token with S.  SR: the 16 random bits of logical element i = t * N + n are
 * bits [16*(i&1), 16*(i&1)+16) of word (i>>1)&3 of Philox4x32-10(key = sr_seed,
 * ctr = (i>>3 low, i>>3 high, 0, 0)); with a = |x*r| < 6 between grid points lo < hi, the code
 * rounds up iff (a - lo)/(hi - lo) > bits * 2^-16.
 *   x [T, N] BF16
 *   colwise = 1: q [N, T/2], s mx_scale_bytes(N, T, 16); requires T % 16 == 0, N % 8 == 0,
 *                T <= 65535 * 128 (grid limit)
 *   colwise = 0: q [T, N/2], s mx_scale_bytes(T, N, 16); requires N % 16 == 0; rht must be 0
 *   s_tensor: one FP32 (written);  workspace: mx_workspace_bytes(MX_WS_1X16, 0, 0) bytes. */
mx_status mx_nvfp4_quantize_1x16(const void* x, int64_t T, int64_t N, int colwise, int rht,
                                 uint64_t rht_seed, mx_round rnd, uint64_t sr_seed,
                                 uint8_t* q, uint8_t* s, float* s_tensor,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Dequantize codes + scales to BF16 (the "dequantized backward" operand DQ(Q(w))).
 * Source: NVFP4 RL page, "dequantized backward" -- y = x * DQ(Q(w_bf16)) rebuilds BF16 operands
 * from the exact low-precision forward values; Miles page (high-precision vs dequantized backward).
 *   MXFP8: y = BF16 RNE of val(q) * 2^(s - 127);  q [rows, cols]; s mx_scale_bytes(rows, cols, 32);
 *          s2 ignored.
 *   NVFP4: y = BF16 RNE of fp32(val(q) * val(bs)) * S; q [rows, cols/2]; s mx_scale_bytes(rows, cols,
 *          16); S = s2[row] (MX_SCOPE_ROW), s2[row / group_rows] (MX_SCOPE_GROUP: stacked matrices of
 *          group_rows rows each, e.g. per-expert 2D weights; group_rows % 128 == 0 so the stacked scale
 *          tensors form one layout) or s2[0] (MX_SCOPE_TENSOR).
 *   y [rows, cols] BF16.  Requires cols % 32 (MXFP8) or cols % 16 (NVFP4) == 0. */
mx_status mx_dequantize_bf16(mx_format fmt, const uint8_t* q, const uint8_t* s, const float* s2,
                             mx_scope s2_scope, int64_t group_rows, int64_t rows, int64_t cols, void* y,
                             cudaStream_t stream);

/* Block-scaled GEMM on the 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA operand
 * staging):  D[m, n] = BF16( alpha_a[m or 0] * alpha_b[n or 0] * sum_k DQ(A)[m, k] * DQ(B)[n, k] ).
 * Source: Miles page -- MXFP8 forward, weight-gradient and data-gradient GEMMs; MaxText page -- the
 * FPROP, DGRAD and WGRAD GEMMs take NVFP4 inputs and emit BF16; E2E page Table 6 (GEMM time).
 * FPROP: A = X row-wise, B = W row-wise.  DGRAD: A = dY row-wise, B = W column-wise.  WGRAD:
 * A = dY column-wise, B = X column-wise.
 *   fmt MX_FMT_MXFP8: a [M, K], b [N, K] E4M3; sa mx_scale_bytes(M, K, 32), sb (N, K, 32).
 *   fmt MX_FMT_NVFP4: a [M, K/2], b [N, K/2] E2M1; sa mx_scale_bytes(M, K, 16), sb (N, K, 16).
 *   alpha_a: NULL / MX_SCOPE_NONE (1), one FP32 (MX_SCOPE_TENSOR) or M FP32 (MX_SCOPE_ROW); alpha_b
 *   likewise with N.  d [M, ldd] BF16.
 * FP32 accumulation inside the tensor core; the summation order is the hardware's.  Requires
 * K % 128 (MXFP8) or K % 256 (NVFP4) == 0; M, N >= 1; N % 8 == 0 and ldd % 8 == 0 (d is written by
 * TMA tensor stores, whose row pitch is a multiple of 16 bytes), ldd >= N; a, b, sa, sb, d 16-byte
 * aligned.  Runs as persistent clusters of two CTAs (one per SM) on 256 x 256 output tiles; large
 * dense MXFP8 GEMMs without a per-column alpha_b take 256 x 384 tiles where the tile count fills the
 * GPU's CTA pairs at least as evenly. */
mx_status mx_scaled_gemm(mx_format fmt,
                         const uint8_t* a, const uint8_t* sa, const float* alpha_a, mx_scope alpha_a_scope,
                         const uint8_t* b, const uint8_t* sb, const float* alpha_b, mx_scope alpha_b_scope,
                         int64_t M, int64_t N, int64_t K, void* d, int64_t ldd, cudaStream_t stream);

/* BF16 GEMM with a dequantized-NVFP4 B operand expanded inside the GEMM (the "dequantized backward"
 * without a BF16 copy of B in HBM):
 *   D[m, n] = BF16( alpha_a[m or 0] * sum_k A[m, k] * DQ(B)[n, k] ),
 *   DQ(B)[n, k] = BF16( fp32(val(q) * val(bs)) * S ), the values mx_dequantize_bf16 writes for B.
 * Source: 4-bitter page, "dequantized backward" -- the backward GEMMs use BF16 operands rebuilt from the
 * forward's exact NVFP4 values (y = x * DQ(Q(w))), which cut the peak memory by 70 % (150 -> 45 MB for a
 * 2k x 2k input and 8k output features); MaxText page (2D weight blocks give the same values in the FPROP
 * and DGRAD orientations).  Data gradient of a linear layer: A = dY [T, O] BF16, B = the column-wise codes
 * of the 2D-quantized weight [H, O/2] with their scales and S_w, D = dX [T, H].
 *   a      [M, K] BF16, contiguous (row pitch K)
 *   alpha_a NULL / MX_SCOPE_NONE, one FP32 (MX_SCOPE_TENSOR) or M FP32 (MX_SCOPE_ROW)
 *   qb     [N, K/2] E2M1 codes (even element in the low nibble); sb mx_scale_bytes(N, K, 16) E4M3 scales
 *          in the GEMM layout; sb2 the FP32 second-level scale: one value (MX_SCOPE_TENSOR) or one per B
 *          row (MX_SCOPE_ROW)
 *   d      [M, ldd] BF16
 * FP32 accumulation in the tensor core (kind::f16), summation order the hardware's.  Requires K % 64 == 0,
 * N % 8 == 0, ldd % 8 == 0, ldd >= N, M, N < 2^31; a, qb, sb, d 16-byte aligned.  Persistent clusters of
 * two CTAs on 512 x 256 output tiles (two M = 256 pair MMAs per K step share each expanded B tile). */
mx_status mx_gemm_bf16_dq_nvfp4(const void* a, const float* alpha_a, mx_scope alpha_a_scope, const uint8_t* qb,
                                const uint8_t* sb, const float* sb2, mx_scope sb2_scope, int64_t M, int64_t N,
                                int64_t K, void* d, int64_t ldd, cudaStream_t stream);

/* Weight gradient of the dequantized backward, X's NVFP4 codes expanded inside the GEMM:
 *   dW[o, h] = BF16( sum_t dY[t, o] * DQ(X)[t, h] ),  DQ(X)[t, h] = BF16( fp32(val(q) * val(bs)) * S ),
 * the values mx_dequantize_bf16 writes for X quantized 1x16 along h (per-token S: MX_SCOPE_ROW, one S per
 * token row; per-tensor: MX_SCOPE_TENSOR).  Both operands are read as stored (tokens along K, neither
 * transposed): dY through 64 x 64 TMA boxes into MN-major tiles, X's codes expanded into MN-major BF16 tiles.
 * Source: 4-bitter page, "dequantized backward" (the backward GEMMs run on BF16 operands rebuilt from the
 * forward's exact NVFP4 values).
 *   dy     [T, O] BF16, contiguous
 *   qx     [T, H/2] E2M1 codes; sx mx_scale_bytes(T, H, 16) E4M3 scales in the GEMM layout; sx2 T FP32
 *          (MX_SCOPE_ROW) or one FP32 (MX_SCOPE_TENSOR)
 *   dw     [O, ldd] BF16
 * FP32 accumulation in the tensor core.  Requires T % 64 == 0, H % 32 == 0, ldd % 8 == 0, ldd >= H,
 * O, H < 2^31; dy, qx, sx, dw 16-byte aligned. */
mx_status mx_wgrad_bf16_dq_nvfp4(const void* dy, const uint8_t* qx, const uint8_t* sx, const float* sx2,
                                 mx_scope sx2_scope, int64_t T, int64_t O, int64_t H, void* dw, int64_t ldd,
                                 cudaStream_t stream);

/* Blockwise FP8 GEMM with FP32 scales (the DeepSeek-V3 form):
 *   D[m, n] = BF16( sum_kb sa[m, kb] * sb[n / 128, kb] * sum_{k in kb} A[m, k] * B[n, k] ),  kb = k / 128
 * Source: NeMo RL FP8 page, "FP8 nas camadas lineares" -- [1, 128] activation / gradient tiles and [128, 128]
 * weight blocks, each with an FP32 scale (the DeepSeek-V3 recipe); E2E page Table 1 -- with FP32 scales (as
 * opposed to power-of-two ones) the scaling runs around the tensor cores on SM100.  Each 128-deep K block
 * is multiplied on the tensor cores (E4M3, FP32 accumulation) and promoted into FP32 accumulators with its
 * scale product.  Forward: A = X row-wise codes with their [R, K/128] scales, B = W's row-wise codes of the
 * [128, 128] quantizer with its block scales s; data gradient: A = dY row-wise, B = W's column-wise codes with
 * the transposed block-scale matrix (sᵀ).
 *   a  [M, K] E4M3, sa [M, K/128] FP32;  b [N, K] E4M3, sb [ceil(N/128), K/128] FP32;  d [M, ldd] BF16
 * Requires K % 128 == 0, N % 8 == 0, ldd % 8 == 0, ldd >= N; a, b, d 16-byte aligned, sa and sb 4-byte
 * aligned.  Persistent clusters of two CTAs on 256 x 256 tiles. */
mx_status mx_fp8_blockwise_gemm(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb, int64_t M,
                                int64_t N, int64_t K, void* d, int64_t ldd, cudaStream_t stream);

/* Blockwise FP8 weight-gradient GEMM with FP32 scales: both operands are contracted over tokens, so both
 * are the column-wise [1, 128] copies of mx_fp8_blockwise_quantize_1x128 (tiles along K = tokens), each
 * row with its own FP32 scale per 128-token block:
 *   D[m, n] = BF16( sum_kb sa[m, kb] * sb[n, kb] * sum_{k in kb} A[m, k] * B[n, k] ),   kb = k / 128
 * e.g. dW [O, H] = dY^T X with A = dY's q_col [O, T], sa = its s_col [O, T/128], B = X's q_col [H, T],
 * sb = its s_col [H, T/128].
 * Source: NeMo RL FP8 page, "FP8 nas camadas lineares" -- input activations and output gradients in
 * [1, 128] tiles with an FP32 scale each (the DeepSeek-V3 recipe), which the weight gradient consumes along
 * tokens; E2E page Table 1 -- FP32 scales are applied around the tensor cores on SM100.
 *   a [M, K] E4M3, sa [M, K/128] FP32;  b [N, K] E4M3, sb [N, K/128] FP32;  d [M, ldd] BF16
 * Requirements as mx_fp8_blockwise_gemm. */
mx_status mx_fp8_blockwise_gemm_wgrad(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb, int64_t M,
                                      int64_t N, int64_t K, void* d, int64_t ldd, cudaStream_t stream);

/* Grouped block-scaled GEMM over expert-sorted rows: for every group g,
 *   D[rows of g] = BF16( alpha_a[row] * alpha_b[g] * A[rows of g] . B_g^T ).
 * Source: Miles page -- NVFP4 on the routed experts' weights and activations with a per-token
 * scale; E2E page Table 2 (Qwen3-30B-A3B: 128 experts, top-8).
 *   group_offsets: DEVICE int64 [G + 1], nondecreasing, offsets[0] = 0, offsets[G] = total_rows;
 *   1 <= G <= MX_MAX_GROUPS.
 *   a [total_rows, K(/2)] codes in plain row order; sa in the grouped scale layout
 *   (mx_grouped_scale_bytes(total_rows, G, K, block), as written by the *_grouped quantizers);
 *   alpha_a_rows [total_rows] FP32 or NULL;  b [G, N, K(/2)], sb G * mx_scale_bytes(N, K, block),
 *   alpha_b_groups [G] FP32 or NULL;  d [total_rows, N] BF16.
 * Same K rules as mx_scaled_gemm; N % 8 == 0. */
mx_status mx_grouped_scaled_gemm(mx_format fmt, int64_t G, const int64_t* group_offsets,
                                 int64_t total_rows,
                                 const uint8_t* a, const uint8_t* sa, const float* alpha_a_rows,
                                 const uint8_t* b, const uint8_t* sb, const float* alpha_b_groups,
                                 int64_t N, int64_t K, void* d, cudaStream_t stream);

/* Count differing bytes between x and y (the offline byte comparison of synchronized weights).
 * Source: E2E page abstract ("synchronized weights ... equal the learner's FP8 forward weights byte
 * for byte") and Table 11 (byte comparison check).
 * Adds the number of positions i < nbytes with x[i] != y[i] to *count (a DEVICE uint64 that the
 * caller zeroes).  x and y 16-byte aligned. */
mx_status mx_count_mismatch(const uint8_t* x, const uint8_t* y, int64_t nbytes,
                            unsigned long long* count, cudaStream_t stream);

/* The weight-sync sweep (E2E page abstract and Table 11: synchronized weights quantized to MXFP8 and
 * NVFP4-2D, dequantized and re-quantized, compared byte for byte) reads each weight stack for its
 * MXFP8 quantization and again, twice, for the NVFP4 2D quantization (whose per-matrix second-level
 * scale needs the matrix maximum first).  These three calls carry that maximum from the pass that
 * already reads the values to the 2D quantizer, which then reads the weights once.  Maxima are
 * 32-bit words holding the BF16 bits of max |x| in the high half (low half zero); DEVICE arrays of
 * one word per matrix, written (not accumulated) by the producing call.
 *
 * mx_quantize_mxfp8 of a stack of matrices [rows = G * matrix_rows, cols], row-wise output required
 * (column-wise optional), plus amax[g] = max |x| over matrix g.  matrix_rows % 128 == 0 and
 * rows % matrix_rows == 0; otherwise the rules of mx_quantize_mxfp8. */
mx_status mx_quantize_mxfp8_amax(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                 uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                 int64_t matrix_rows, uint32_t* amax, cudaStream_t stream);

/* mx_nvfp4_quantize_weight_2d with each matrix's maximum supplied (amax[g], as above) instead of
 * measured: identical results when amax[g] is the true max |w_g|, and one read of the weights. */
mx_status mx_nvfp4_quantize_weight_2d_given_amax(const void* w, int64_t G, int64_t O, int64_t H,
                                                 uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                                                 uint8_t* s_col, float* s_w, const uint32_t* amax,
                                                 cudaStream_t stream);

/* mx_dequantize_bf16 of NVFP4 with one second-level scale per group of group_rows rows
 * (MX_SCOPE_GROUP), plus amax[g] = max |y| over group g of the BF16 output.  group_rows % 128 == 0,
 * rows % group_rows == 0, cols % 16 == 0. */
mx_status mx_dequantize_nvfp4_amax(const uint8_t* q, const uint8_t* s, const float* s2, int64_t group_rows,
                                   int64_t rows, int64_t cols, void* y, uint32_t* amax, cudaStream_t stream);

/* Workspace sizes (bytes) for the ops that take one. */
typedef enum { MX_WS_WEIGHT_2D = 0, MX_WS_1X16 = 1 } mx_workspace_op;
size_t mx_workspace_bytes(mx_workspace_op op, int64_t groups, int64_t unused);

/* Failure detection.  Every mbarrier wait inside the kernels is bounded (2 s): a wait that gives up
 * sets a device-side watchdog word (one per kernel family: the GEMMs, the MXFP8 quantizer), stops
 * its CTA from issuing more work, lets the copies already issued land, and the CTA exits; its
 * outputs are then undefined.  The calls below report and clear those words.
 * Source: the E2E page, Tables 11-13 (the checks a low-precision RL run keeps and the faults each
 * catches); the pages describe the failures, not this mechanism.
 *
 * mx_check_device_status: synchronizes the device, then returns MX_ERR_TIMEOUT if any watchdog word
 * is set (and clears them all), MX_ERR_CUDA if the device reports an error, else MX_OK. */
mx_status mx_check_device_status(void);

/* As mx_check_device_status, waiting for `stream` only: the words are read and cleared by copies
 * ordered on `stream`, then the stream is synchronized.  The words are shared by every stream of
 * the device, so a timeout recorded by work on another stream is reported (and cleared) here too. */
mx_status mx_check_stream_status(cudaStream_t stream);

/* Watchdog self-test (test hook).  Launches, on `stream`, one small kernel of the chosen family
 * whose waits are on barriers nothing ever arrives on, each bounded by `limit_ns` instead of the
 * kernels' 2 s: MX_WATCHDOG_GEMM runs a cluster of two CTAs set up as the pair GEMMs are (TMEM
 * allocated for the pair) and leaves through their exit path; MX_WATCHDOG_MXFP8 runs one CTA of
 * waits on the MXFP8 quantizer's word.  No copy or MMA is issued, so the expiry is the only fault.
 * Afterwards mx_check_device_status / mx_check_stream_status return MX_ERR_TIMEOUT once, then MX_OK.
 *   limit_ns in [1000, 1000000000], else MX_ERR_INVALID_ARG. */
typedef enum { MX_WATCHDOG_GEMM = 0, MX_WATCHDOG_MXFP8 = 1 } mx_watchdog_unit;
mx_status mx_watchdog_selftest(mx_watchdog_unit unit, uint64_t limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MXNUM_H */
