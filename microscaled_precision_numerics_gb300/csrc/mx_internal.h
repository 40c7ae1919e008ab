// mx_internal.h -- declarations shared by the mxnum translation units (not part of the C ABI).
#pragma once

#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "mx_device.cuh"

namespace mxk {

// Division of an unsigned 32-bit n by an invariant d >= 1 with one multiply-high, after Granlund and
// Montgomery, "Division by invariant integers using multiplication" (PLDI 1994), section 4:
// l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1, and q = (t + ((n - t) >> s1)) >> s2 with
// t = mulhi(m, n), s1 = min(l, 1), s2 = max(l - 1, 0); exact for every n < 2^32.
struct DivU32 {
    uint32_t m, s1, s2;
};
inline DivU32 make_divu32(uint64_t d) {
    uint32_t l = 0;
    while (l < 32 && (1ull << l) < d) ++l;
    const uint64_t m = (((1ull << l) - d) << 32) / d + 1;
    return DivU32{(uint32_t)m, l > 0 ? 1u : 0u, l > 0 ? l - 1 : 0u};
}
__device__ __forceinline__ uint32_t divu32(uint32_t n, DivU32 d) {
    const uint32_t t = __umulhi(n, d.m);
    return (t + ((n - t) >> d.s1)) >> d.s2;
}

// One-time setup per device: kernel attributes (and the occupancy read after them) belong to each
// device's context, so a process that drives several GPUs sets them once on every device.  The first
// call with a device current runs f(value), which returns a CUDA status and may store one integer.
constexpr int MX_MAX_DEVICES = 64;
struct PerDevice {
    std::once_flag once[MX_MAX_DEVICES];
    cudaError_t err[MX_MAX_DEVICES] = {};
    int value[MX_MAX_DEVICES] = {};
};
template <typename F>
inline cudaError_t per_device_once(PerDevice& pd, int& value, F&& f) {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MX_MAX_DEVICES) return cudaErrorInvalidDevice;
    std::call_once(pd.once[dev], [&] { pd.err[dev] = f(pd.value[dev]); });
    value = pd.value[dev];
    return pd.err[dev];
}

// Grid limits (grid y and z are at most 65535): the 2D weight quantizer launches one grid row per
// W2D_TILE_ROWS matrix rows and one grid layer per matrix, the column-wise 1x16 quantizer one grid row
// per CW_TILE_TOKENS tokens.  The entry points refuse larger shapes.
constexpr int64_t MX_GRID_YZ_MAX = 65535;
constexpr int W2D_TILE_ROWS = 64;
constexpr int CW_TILE_TOKENS = 128;
inline bool weight_2d_grid_ok(int64_t G, int64_t O) {
    return G <= MX_GRID_YZ_MAX && (O + W2D_TILE_ROWS - 1) / W2D_TILE_ROWS <= MX_GRID_YZ_MAX;
}
inline bool colwise_grid_ok(int64_t T) { return (T + CW_TILE_TOKENS - 1) / CW_TILE_TOKENS <= MX_GRID_YZ_MAX; }

// Bytes of a GEMM-layout scale tensor (see include/mxnum.h).
__host__ __device__ inline int64_t host_scale_bytes(int64_t rows, int64_t k, int block) {
    return ((rows + 127) / 128) * ((k / block + 3) / 4) * 512;
}
__host__ __device__ inline int64_t host_scale_bytes_dev(int64_t rows, int64_t k, int block) {
    return host_scale_bytes(rows, k, block);
}

// RHT sign mask computed on the host with the same Philox4x32-10 definition as the device.
uint32_t host_rht_sign_mask(uint64_t seed);

// One tensor of an MXFP8 quantize launch (null q_row / q_col: that orientation is skipped).
struct Mx8Tensor {
    const uint16_t* x;
    int64_t R, K, ldx;
    uint8_t *q_row, *s_row, *q_col, *s_col;
};
constexpr int MX8_MAX_BATCH = 4;
// Several tensors in one launch; all of them must request the same orientations.
cudaError_t launch_mxfp8_quantize_batched(const Mx8Tensor* ts, int n, cudaStream_t stream);
// One tensor of stacked matrices (matrix_rows rows each, a multiple of 128), row-wise output required;
// also writes each matrix's max |x| (BF16 bits << 16) to amax.
cudaError_t launch_mxfp8_quantize_amax(const Mx8Tensor& t, int64_t matrix_rows, uint32_t* amax, cudaStream_t stream);
cudaError_t launch_mxfp8_quantize(const uint16_t* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q_row,
                                  uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, int G, const int64_t* group_offsets,
                                  cudaStream_t stream);
cudaError_t launch_nvfp4_per_token(const uint16_t* x, int64_t T, int64_t H, int64_t ldx, uint8_t* q, uint8_t* s,
                                   float* s_tok, int G, const int64_t* group_offsets, int num_sms, cudaStream_t stream,
                                   bool four_six = false);
cudaError_t launch_nvfp4_1x16(const uint16_t* x, int64_t T, int64_t N, bool colwise, bool rht, uint64_t rht_seed,
                              bool sr, uint64_t sr_seed, uint8_t* q, uint8_t* s, float* s_tensor, uint32_t* ws,
                              int num_sms, cudaStream_t stream);
cudaError_t launch_rht16(const uint16_t* x, int64_t T, int64_t N, uint64_t seed, uint16_t* y, cudaStream_t stream);
cudaError_t launch_nvfp4_weight_2d(const uint16_t* w, int64_t G, int64_t O, int64_t H, uint8_t* q_row, uint8_t* s_row,
                                   uint8_t* q_col, uint8_t* s_col, float* s_w, uint32_t* ws, int num_sms,
                                   cudaStream_t stream, bool four_six = false);
cudaError_t launch_fp8_blockwise_1x128(const uint16_t* x, int64_t R, int64_t K, int64_t ldx, bool pow2,
                                       uint8_t* q_row, float* s_row, uint8_t* sf_row, uint8_t* q_col, float* s_col,
                                       uint8_t* sf_col, int num_sms, cudaStream_t stream);
cudaError_t launch_fp8_blockwise_128x128(const uint16_t* w, int64_t G, int64_t O, int64_t H, bool pow2,
                                         uint8_t* q_row, uint8_t* q_col, float* s, uint8_t* sf_row, uint8_t* sf_col,
                                         int num_sms, cudaStream_t stream);
cudaError_t launch_dequant(int fmt, const uint8_t* q, const uint8_t* s, const float* s2, int64_t rows_per_scale, int64_t R,
                           int64_t K, uint16_t* y, cudaStream_t stream);
cudaError_t launch_mismatch(const uint8_t* x, const uint8_t* y, int64_t nbytes, unsigned long long* count,
                            int num_sms, cudaStream_t stream);

// Block-scaled tcgen05 GEMM (dense and grouped).  fmt: 0 MXFP8, 1 NVFP4.  alpha scopes: 0 none,
// 1 tensor, 2 row (per M row for a, per N column for b; per group for grouped b).
struct GemmArgs {
    int fmt;
    const uint8_t* a; const uint8_t* sa; const float* alpha_a; int alpha_a_scope;
    const uint8_t* b; const uint8_t* sb; const float* alpha_b; int alpha_b_scope;
    int64_t M, N, K;
    uint16_t* d; int64_t ldd;
    // grouped: G > 0 and group_offsets (device) describe the expert-sorted row groups of a; b holds G
    // matrices [N, K] with per-group scale tensors; alpha_b is per group.
    int64_t G; const int64_t* group_offsets;
};
cudaError_t launch_scaled_gemm(const GemmArgs& args, int num_sms, cudaStream_t stream);

// BF16 x dequantized-NVFP4 GEMM.  K-major form: A BF16 [M, K]; B NVFP4 codes [N, K/2], E4M3 scales in the GEMM
// layout and an FP32 second-level scale (sb2_scope 1: one value, 2: per B row).  Weight-gradient form
// (wgrad): A BF16 [K, M] (dY), B codes [K, N/2] with scales (K, N, 16) (X quantized along N) and sb2_scope
// 1 or 3 (per K row, i.e. per token); D = A^T DQ(B).  alpha_a as in GemmArgs.
struct DqGemmArgs {
    const uint16_t* a; const float* alpha_a; int alpha_a_scope;
    const uint8_t* qb; const uint8_t* sb; const float* sb2; int sb2_scope;
    int64_t M, N, K;
    uint16_t* d; int64_t ldd;
    bool wgrad;
};
cudaError_t launch_dq_gemm(const DqGemmArgs& args, int num_sms, cudaStream_t stream);

// Blockwise FP8 GEMM with FP32 scales: a [M, K] and b [N, K] E4M3 (K-major); sa [M, K/128] FP32 (one per
// [1, 128] tile of a), sb [ceil(N/128), K/128] FP32 (one per [128, 128] block of b).
struct BwGemmArgs {
    const uint8_t* a; const float* sa; const uint8_t* b; const float* sb;
    int64_t M, N, K;
    uint16_t* d; int64_t ldd;
    bool b_row_scales;        // sb [N, K/128] (one scale per B row) instead of [ceil(N/128), K/128]
};
cudaError_t launch_fp8_blockwise_gemm(const BwGemmArgs& args, int num_sms, cudaStream_t stream);
cudaError_t launch_nvfp4_weight_2d_given_amax(const uint16_t* w, int64_t G, int64_t O, int64_t H, uint8_t* q_row,
                                              uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, float* s_w,
                                              const uint32_t* amax, cudaStream_t stream);
cudaError_t launch_dequant_nvfp4_amax(const uint8_t* q, const uint8_t* s, const float* s2, int64_t group_rows, int64_t R,
                                      int64_t K, uint16_t* y, uint32_t* amax, cudaStream_t stream);
uint32_t read_and_clear_device_status();
uint32_t read_and_clear_mxfp8_status();
uint32_t read_and_clear_device_status_on(cudaStream_t stream);
uint32_t read_and_clear_mxfp8_status_on(cudaStream_t stream);
cudaError_t launch_watchdog_selftest(unsigned long long limit_ns, cudaStream_t stream);
cudaError_t launch_mxfp8_watchdog_selftest(unsigned long long limit_ns, cudaStream_t stream);

int device_sm_count();

}  // namespace mxk
