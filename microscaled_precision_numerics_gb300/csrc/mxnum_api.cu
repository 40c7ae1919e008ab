// mxnum_api.cu -- the C ABI of libmxnum.so: argument validation and launches (see include/mxnum.h).
#include "../../include/mxnum.h"
#include "mx_internal.h"

#include <mutex>

namespace mxk {

uint32_t host_rht_sign_mask(uint64_t seed) {
    // Philox4x32-10 with key = seed, counter = (0, 0, 1, 0); bits 0..15 of word 0.
    uint32_t c0 = 0, c1 = 0, c2 = 1, c3 = 0;
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    for (int rnd = 0; rnd < 10; ++rnd) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0, p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0, n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        c0 = n0; c1 = (uint32_t)p1; c2 = n2; c3 = (uint32_t)p0;
        k0 += 0x9E3779B9u; k1 += 0xBB67AE85u;
    }
    return c0 & 0xFFFFu;
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

}  // namespace mxk

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline mx_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MX_OK : MX_ERR_CUDA; }

}  // namespace

extern "C" {

const char* mx_status_string(mx_status s) {
    switch (s) {
        case MX_OK: return "MX_OK";
        case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG";
        case MX_ERR_ALIGNMENT: return "MX_ERR_ALIGNMENT";
        case MX_ERR_UNSUPPORTED: return "MX_ERR_UNSUPPORTED";
        case MX_ERR_CUDA: return "MX_ERR_CUDA";
        case MX_ERR_TIMEOUT: return "MX_ERR_TIMEOUT";
    }
    return "MX_ERR_UNKNOWN";
}

int64_t mx_scale_bytes(int64_t rows, int64_t k, int block) {
    if (rows <= 0 || k <= 0 || (block != 16 && block != 32)) return 0;
    return mxk::host_scale_bytes(rows, k, block);
}

size_t mx_workspace_bytes(mx_workspace_op op, int64_t groups, int64_t /*unused*/) {
    switch (op) {
        case MX_WS_WEIGHT_2D: return groups > 0 ? (size_t)(((groups * 4) + 15) / 16 * 16) : 0;
        case MX_WS_1X16: return 16;
    }
    return 0;
}

static mx_status check_mxfp8_args(const void* x, int64_t rows, int64_t cols, int64_t ldx, const uint8_t* q_row,
                                  const uint8_t* s_row, const uint8_t* q_col, const uint8_t* s_col) {
    if (!x || rows <= 0 || cols <= 0 || ldx < cols) return MX_ERR_INVALID_ARG;
    if (!q_row && !q_col) return MX_ERR_INVALID_ARG;
    if ((q_row && !s_row) || (q_col && !s_col)) return MX_ERR_INVALID_ARG;
    if ((cols % 8) != 0 || (ldx % 8) != 0) return MX_ERR_ALIGNMENT;
    if (!aligned16(x) || (q_row && (!aligned16(q_row) || !aligned16(s_row))) ||
        (q_col && (!aligned16(q_col) || !aligned16(s_col))))
        return MX_ERR_ALIGNMENT;
    if (q_row && (cols % 32) != 0) return MX_ERR_UNSUPPORTED;
    if (q_col && (rows % 32) != 0) return MX_ERR_UNSUPPORTED;
    return MX_OK;
}

mx_status mx_quantize_mxfp8(const void* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q_row, uint8_t* s_row,
                            uint8_t* q_col, uint8_t* s_col, cudaStream_t stream) {
    const mx_status st = check_mxfp8_args(x, rows, cols, ldx, q_row, s_row, q_col, s_col);
    if (st != MX_OK) return st;
    return from_cuda(mxk::launch_mxfp8_quantize(static_cast<const uint16_t*>(x), rows, cols, ldx, q_row, s_row,
                                                 q_col, s_col, 0, nullptr, stream));
}

mx_status mx_quantize_mxfp8_amax(const void* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q_row, uint8_t* s_row,
                                 uint8_t* q_col, uint8_t* s_col, int64_t matrix_rows, uint32_t* amax, cudaStream_t stream) {
    const mx_status st = check_mxfp8_args(x, rows, cols, ldx, q_row, s_row, q_col, s_col);
    if (st != MX_OK) return st;
    if (!q_row || !amax || matrix_rows <= 0) return MX_ERR_INVALID_ARG;
    if (!aligned16(amax)) return MX_ERR_ALIGNMENT;
    if ((matrix_rows % 128) != 0 || (rows % matrix_rows) != 0) return MX_ERR_UNSUPPORTED;
    const mxk::Mx8Tensor t{static_cast<const uint16_t*>(x), rows, cols, ldx, q_row, s_row, q_col, s_col};
    return from_cuda(mxk::launch_mxfp8_quantize_amax(t, matrix_rows, amax, stream));
}

mx_status mx_quantize_mxfp8_batched(const mx_mxfp8_tensor* tensors, int count, cudaStream_t stream) {
    static_assert(MX_MXFP8_MAX_BATCH == mxk::MX8_MAX_BATCH, "batch limit");
    if (!tensors || count < 1 || count > MX_MXFP8_MAX_BATCH) return MX_ERR_INVALID_ARG;
    mxk::Mx8Tensor ts[MX_MXFP8_MAX_BATCH];
    for (int i = 0; i < count; ++i) {
        const mx_mxfp8_tensor& t = tensors[i];
        const mx_status st = check_mxfp8_args(t.x, t.rows, t.cols, t.ldx, t.q_row, t.s_row, t.q_col, t.s_col);
        if (st != MX_OK) return st;
        if ((t.q_row != nullptr) != (tensors[0].q_row != nullptr) || (t.q_col != nullptr) != (tensors[0].q_col != nullptr))
            return MX_ERR_INVALID_ARG;
        ts[i] = mxk::Mx8Tensor{static_cast<const uint16_t*>(t.x), t.rows, t.cols, t.ldx, t.q_row, t.s_row, t.q_col, t.s_col};
    }
    return from_cuda(mxk::launch_mxfp8_quantize_batched(ts, count, stream));
}

mx_status mx_quantize_mxfp8_grouped(const void* x, int64_t rows, int64_t cols, int64_t ldx, int64_t G,
                                    const int64_t* group_offsets, uint8_t* q_row, uint8_t* s_row, cudaStream_t stream) {
    if (!x || !q_row || !s_row || !group_offsets || rows <= 0 || cols <= 0 || ldx < cols) return MX_ERR_INVALID_ARG;
    if (G <= 0 || G > MX_MAX_GROUPS) return MX_ERR_INVALID_ARG;
    if ((cols % 8) != 0 || (ldx % 8) != 0 || !aligned16(x) || !aligned16(q_row) || !aligned16(s_row) ||
        !aligned16(group_offsets))
        return MX_ERR_ALIGNMENT;
    if ((cols % 32) != 0) return MX_ERR_UNSUPPORTED;
    return from_cuda(mxk::launch_mxfp8_quantize(static_cast<const uint16_t*>(x), rows, cols, ldx, q_row, s_row,
                                                 nullptr, nullptr, (int)G, group_offsets, stream));
}

int64_t mx_grouped_scale_bytes(int64_t rows, int64_t G, int64_t k, int block) {
    if (rows <= 0 || G <= 0 || k <= 0 || (block != 16 && block != 32)) return 0;
    return mxk::host_scale_bytes(rows + 127 * G, k, block);
}

mx_status mx_nvfp4_quantize_per_token(const void* x, int64_t T, int64_t H, int64_t ldx, uint8_t* q, uint8_t* s,
                                      float* s_tok, cudaStream_t stream) {
    if (!x || !q || !s || !s_tok || T <= 0 || H <= 0 || ldx < H) return MX_ERR_INVALID_ARG;
    if ((ldx % 8) != 0 || !aligned16(x) || !aligned16(q) || !aligned16(s) || !aligned16(s_tok)) return MX_ERR_ALIGNMENT;
    if ((H % 16) != 0) return MX_ERR_UNSUPPORTED;
    return from_cuda(mxk::launch_nvfp4_per_token(static_cast<const uint16_t*>(x), T, H, ldx, q, s, s_tok, 0, nullptr,
                                                  mxk::device_sm_count(), stream));
}

mx_status mx_nvfp4_quantize_per_token_grouped(const void* x, int64_t T, int64_t H, int64_t ldx, int64_t G,
                                              const int64_t* group_offsets, uint8_t* q, uint8_t* s, float* s_tok,
                                              cudaStream_t stream) {
    if (!x || !q || !s || !s_tok || !group_offsets || T <= 0 || H <= 0 || ldx < H) return MX_ERR_INVALID_ARG;
    if (G <= 0 || G > MX_MAX_GROUPS) return MX_ERR_INVALID_ARG;
    if ((ldx % 8) != 0 || !aligned16(x) || !aligned16(q) || !aligned16(s) || !aligned16(s_tok) ||
        !aligned16(group_offsets))
        return MX_ERR_ALIGNMENT;
    if ((H % 16) != 0) return MX_ERR_UNSUPPORTED;
    return from_cuda(mxk::launch_nvfp4_per_token(static_cast<const uint16_t*>(x), T, H, ldx, q, s, s_tok, (int)G,
                                                  group_offsets, mxk::device_sm_count(), stream));
}

mx_status mx_nvfp4_quantize_weight_2d(const void* w, int64_t G, int64_t O, int64_t H, uint8_t* q_row, uint8_t* s_row,
                                      uint8_t* q_col, uint8_t* s_col, float* s_w, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream) {
    if (!w || !q_row || !s_row || !q_col || !s_col || !s_w || !workspace) return MX_ERR_INVALID_ARG;
    if (G <= 0 || O <= 0 || H <= 0) return MX_ERR_INVALID_ARG;
    if (workspace_bytes < mx_workspace_bytes(MX_WS_WEIGHT_2D, G, 0)) return MX_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q_row) || !aligned16(s_row) || !aligned16(q_col) || !aligned16(s_col) ||
        !aligned16(s_w) || !aligned16(workspace))
        return MX_ERR_ALIGNMENT;
    if ((O % 16) != 0 || (H % 16) != 0 || !mxk::weight_2d_grid_ok(G, O)) return MX_ERR_UNSUPPORTED;
    return from_cuda(mxk::launch_nvfp4_weight_2d(static_cast<const uint16_t*>(w), G, O, H, q_row, s_row, q_col, s_col,
                                                  s_w, static_cast<uint32_t*>(workspace), mxk::device_sm_count(),
                                                  stream));
}

mx_status mx_nvfp4_quantize_per_token_46(const void* x, int64_t T, int64_t H, int64_t ldx, uint8_t* q, uint8_t* s,
                                         float* s_tok, cudaStream_t stream) {
    if (!x || !q || !s || !s_tok || T <= 0 || H <= 0 || ldx < H) return MX_ERR_INVALID_ARG;
    if ((ldx % 8) != 0 || !aligned16(x) || !aligned16(q) || !aligned16(s) || !aligned16(s_tok)) return MX_ERR_ALIGNMENT;
    if ((H % 16) != 0) return MX_ERR_UNSUPPORTED;
    return from_cuda(mxk::launch_nvfp4_per_token(static_cast<const uint16_t*>(x), T, H, ldx, q, s, s_tok, 0, nullptr,
                                                  mxk::device_sm_count(), stream, true));
}

mx_status mx_nvfp4_quantize_weight_2d_46(const void* w, int64_t G, int64_t O, int64_t H, uint8_t* q_row, uint8_t* s_row,
                                         uint8_t* q_col, uint8_t* s_col, float* s_w, void* workspace,
                                         size_t workspace_bytes, cudaStream_t stream) {
    if (!w || !q_row || !s_row || !q_col || !s_col || !s_w || !workspace) return MX_ERR_INVALID_ARG;
    if (G <= 0 || O <= 0 || H <= 0) return MX_ERR_INVALID_ARG;
    if (workspace_bytes < mx_workspace_bytes(MX_WS_WEIGHT_2D, G, 0)) return MX_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q_row) || !aligned16(s_row) || !aligned16(q_col) || !aligned16(s_col) ||
        !aligned16(s_w) || !aligned16(workspace))
        return MX_ERR_ALIGNMENT;
    if ((O % 16) != 0 || (H % 16) != 0 || !mxk::weight_2d_grid_ok(G, O)) return MX_ERR_UNSUPPORTED;
    return from_cuda(mxk::launch_nvfp4_weight_2d(static_cast<const uint16_t*>(w), G, O, H, q_row, s_row, q_col, s_col,
                                                  s_w, static_cast<uint32_t*>(workspace), mxk::device_sm_count(),
                                                  stream, true));
}

mx_status mx_fp8_blockwise_quantize_1x128(const void* x, int64_t rows, int64_t cols, int64_t ldx, int pow2,
                                          uint8_t* q_row, float* s_row, uint8_t* sf_row, uint8_t* q_col, float* s_col,
                                          uint8_t* sf_col, cudaStream_t stream) {
    if (!x || rows <= 0 || cols <= 0 || ldx < cols || (pow2 != 0 && pow2 != 1)) return MX_ERR_INVALID_ARG;
    if (!q_row && !q_col) return MX_ERR_INVALID_ARG;
    if ((q_row && !s_row) || (q_col && !s_col)) return MX_ERR_INVALID_ARG;
    if (!pow2 && (sf_row || sf_col)) return MX_ERR_INVALID_ARG;
    if ((sf_row && !q_row) || (sf_col && !q_col)) return MX_ERR_INVALID_ARG;
    if ((ldx % 8) != 0 || !aligned16(x) || (q_row && (!aligned16(q_row) || !aligned16(s_row))) ||
        (q_col && (!aligned16(q_col) || !aligned16(s_col))) || (sf_row && !aligned16(sf_row)) ||
        (sf_col && !aligned16(sf_col)))
        return MX_ERR_ALIGNMENT;
    if ((cols % 16) != 0) return MX_ERR_UNSUPPORTED;
    if (q_row && (cols % 128) != 0) return MX_ERR_UNSUPPORTED;
    if (q_col && ((rows % 128) != 0 || rows / 128 > 65535)) return MX_ERR_UNSUPPORTED;
    if (rows * (cols / 128) >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    return from_cuda(mxk::launch_fp8_blockwise_1x128(static_cast<const uint16_t*>(x), rows, cols, ldx, pow2 != 0, q_row,
                                                      s_row, sf_row, q_col, s_col, sf_col, mxk::device_sm_count(),
                                                      stream));
}

mx_status mx_fp8_blockwise_quantize_128x128(const void* w, int64_t G, int64_t O, int64_t H, int pow2, uint8_t* q_row,
                                            uint8_t* q_col, float* s, uint8_t* sf_row, uint8_t* sf_col,
                                            cudaStream_t stream) {
    if (!w || !q_row || !q_col || !s || G <= 0 || O <= 0 || H <= 0 || (pow2 != 0 && pow2 != 1))
        return MX_ERR_INVALID_ARG;
    if (G > 65535 || (O + 127) / 128 > 65535) return MX_ERR_UNSUPPORTED;
    if (!pow2 && (sf_row || sf_col)) return MX_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q_row) || !aligned16(q_col) || !aligned16(s) || (sf_row && !aligned16(sf_row)) ||
        (sf_col && !aligned16(sf_col)))
        return MX_ERR_ALIGNMENT;
    if ((O % 16) != 0 || (H % 16) != 0) return MX_ERR_UNSUPPORTED;
    if ((sf_row || sf_col) && ((O % 128) != 0 || (H % 128) != 0)) return MX_ERR_UNSUPPORTED;
    return from_cuda(mxk::launch_fp8_blockwise_128x128(static_cast<const uint16_t*>(w), G, O, H, pow2 != 0, q_row,
                                                        q_col, s, sf_row, sf_col, mxk::device_sm_count(), stream));
}

mx_status mx_rht16(const void* x, int64_t T, int64_t N, uint64_t seed, void* y, cudaStream_t stream) {
    if (!x || !y || T <= 0 || N <= 0 || x == y) return MX_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y) || (N % 8) != 0) return MX_ERR_ALIGNMENT;
    if ((T % 16) != 0) return MX_ERR_UNSUPPORTED;
    return from_cuda(mxk::launch_rht16(static_cast<const uint16_t*>(x), T, N, seed, static_cast<uint16_t*>(y), stream));
}

mx_status mx_nvfp4_quantize_1x16(const void* x, int64_t T, int64_t N, int colwise, int rht, uint64_t rht_seed,
                                 mx_round rnd, uint64_t sr_seed, uint8_t* q, uint8_t* s, float* s_tensor,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!x || !q || !s || !s_tensor || !workspace || T <= 0 || N <= 0) return MX_ERR_INVALID_ARG;
    if (rnd != MX_ROUND_RNE && rnd != MX_ROUND_SR) return MX_ERR_INVALID_ARG;
    if (workspace_bytes < mx_workspace_bytes(MX_WS_1X16, 0, 0)) return MX_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(s) || !aligned16(workspace)) return MX_ERR_ALIGNMENT;
    if (colwise) {
        if ((N % 8) != 0) return MX_ERR_ALIGNMENT;
        if ((T % 16) != 0 || !mxk::colwise_grid_ok(T)) return MX_ERR_UNSUPPORTED;
    } else {
        if (rht) return MX_ERR_UNSUPPORTED;
        if ((N % 16) != 0) return MX_ERR_UNSUPPORTED;
    }
    return from_cuda(mxk::launch_nvfp4_1x16(static_cast<const uint16_t*>(x), T, N, colwise != 0, rht != 0, rht_seed,
                                             rnd == MX_ROUND_SR, sr_seed, q, s, s_tensor,
                                             static_cast<uint32_t*>(workspace), mxk::device_sm_count(), stream));
}

mx_status mx_dequantize_bf16(mx_format fmt, const uint8_t* q, const uint8_t* s, const float* s2, mx_scope s2_scope,
                             int64_t group_rows, int64_t rows, int64_t cols, void* y, cudaStream_t stream) {
    if (!q || !s || !y || rows <= 0 || cols <= 0) return MX_ERR_INVALID_ARG;
    if (fmt != MX_FMT_MXFP8 && fmt != MX_FMT_NVFP4) return MX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(y)) return MX_ERR_ALIGNMENT;
    int64_t per = 0;   // rows sharing one second-level scale (0: one for the whole tensor)
    if (fmt == MX_FMT_MXFP8) {
        if ((cols % 32) != 0) return MX_ERR_UNSUPPORTED;
    } else {
        if (!s2) return MX_ERR_INVALID_ARG;
        if (s2_scope == MX_SCOPE_ROW) per = 1;
        else if (s2_scope == MX_SCOPE_GROUP) {
            if (group_rows <= 0) return MX_ERR_INVALID_ARG;
            if ((group_rows % 128) != 0) return MX_ERR_UNSUPPORTED;
            per = group_rows;
        } else if (s2_scope != MX_SCOPE_TENSOR) return MX_ERR_INVALID_ARG;
        if ((cols % 16) != 0) return MX_ERR_UNSUPPORTED;
    }
    return from_cuda(mxk::launch_dequant(fmt == MX_FMT_MXFP8 ? 0 : 1, q, s, s2, per, rows, cols,
                                         static_cast<uint16_t*>(y), stream));
}

mx_status mx_nvfp4_quantize_weight_2d_given_amax(const void* w, int64_t G, int64_t O, int64_t H, uint8_t* q_row,
                                                 uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, float* s_w,
                                                 const uint32_t* amax, cudaStream_t stream) {
    if (!w || !q_row || !s_row || !q_col || !s_col || !s_w || !amax) return MX_ERR_INVALID_ARG;
    if (G <= 0 || O <= 0 || H <= 0) return MX_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q_row) || !aligned16(s_row) || !aligned16(q_col) || !aligned16(s_col) ||
        !aligned16(s_w) || !aligned16(amax))
        return MX_ERR_ALIGNMENT;
    if ((O % 16) != 0 || (H % 16) != 0 || !mxk::weight_2d_grid_ok(G, O)) return MX_ERR_UNSUPPORTED;
    return from_cuda(mxk::launch_nvfp4_weight_2d_given_amax(static_cast<const uint16_t*>(w), G, O, H, q_row, s_row,
                                                            q_col, s_col, s_w, amax, stream));
}

mx_status mx_dequantize_nvfp4_amax(const uint8_t* q, const uint8_t* s, const float* s2, int64_t group_rows,
                                   int64_t rows, int64_t cols, void* y, uint32_t* amax, cudaStream_t stream) {
    if (!q || !s || !s2 || !y || !amax || rows <= 0 || cols <= 0 || group_rows <= 0) return MX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(y) || !aligned16(amax)) return MX_ERR_ALIGNMENT;
    if ((cols % 16) != 0 || (group_rows % 128) != 0 || (rows % group_rows) != 0) return MX_ERR_UNSUPPORTED;
    return from_cuda(mxk::launch_dequant_nvfp4_amax(q, s, s2, group_rows, rows, cols, static_cast<uint16_t*>(y), amax,
                                                    stream));
}

static mx_status validate_gemm_common(mx_format fmt, const uint8_t* a, const uint8_t* sa, const uint8_t* b,
                                      const uint8_t* sb, int64_t N, int64_t K, const void* d) {
    if (fmt != MX_FMT_MXFP8 && fmt != MX_FMT_NVFP4) return MX_ERR_INVALID_ARG;
    if (!a || !sa || !b || !sb || !d || N <= 0 || K <= 0) return MX_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(sa) || !aligned16(b) || !aligned16(sb) || !aligned16(d)) return MX_ERR_ALIGNMENT;
    const int64_t kstep = fmt == MX_FMT_MXFP8 ? 128 : 256;
    if ((K % kstep) != 0) return MX_ERR_UNSUPPORTED;
    return MX_OK;
}

mx_status mx_scaled_gemm(mx_format fmt, const uint8_t* a, const uint8_t* sa, const float* alpha_a,
                         mx_scope alpha_a_scope, const uint8_t* b, const uint8_t* sb, const float* alpha_b,
                         mx_scope alpha_b_scope, int64_t M, int64_t N, int64_t K, void* d, int64_t ldd,
                         cudaStream_t stream) {
    mx_status st = validate_gemm_common(fmt, a, sa, b, sb, N, K, d);
    if (st != MX_OK) return st;
    if (M <= 0 || ldd < N) return MX_ERR_INVALID_ARG;
    if ((N % 8) != 0 || (ldd % 8) != 0) return MX_ERR_ALIGNMENT;
    if ((alpha_a_scope != MX_SCOPE_NONE && !alpha_a) || (alpha_b_scope != MX_SCOPE_NONE && !alpha_b))
        return MX_ERR_INVALID_ARG;
    if (alpha_a_scope < MX_SCOPE_NONE || alpha_a_scope > MX_SCOPE_ROW || alpha_b_scope < MX_SCOPE_NONE ||
        alpha_b_scope > MX_SCOPE_ROW)
        return MX_ERR_INVALID_ARG;
    mxk::GemmArgs g{};
    g.fmt = fmt == MX_FMT_MXFP8 ? 0 : 1;
    g.a = a; g.sa = sa; g.alpha_a = alpha_a; g.alpha_a_scope = alpha_a ? (int)alpha_a_scope : 0;
    g.b = b; g.sb = sb; g.alpha_b = alpha_b; g.alpha_b_scope = alpha_b ? (int)alpha_b_scope : 0;
    g.M = M; g.N = N; g.K = K; g.d = static_cast<uint16_t*>(d); g.ldd = ldd;
    g.G = 0; g.group_offsets = nullptr;
    return from_cuda(mxk::launch_scaled_gemm(g, mxk::device_sm_count(), stream));
}

mx_status mx_gemm_bf16_dq_nvfp4(const void* a, const float* alpha_a, mx_scope alpha_a_scope, const uint8_t* qb,
                                const uint8_t* sb, const float* sb2, mx_scope sb2_scope, int64_t M, int64_t N,
                                int64_t K, void* d, int64_t ldd, cudaStream_t stream) {
    if (!a || !qb || !sb || !sb2 || !d || M <= 0 || N <= 0 || K <= 0 || ldd < N) return MX_ERR_INVALID_ARG;
    if (alpha_a_scope < MX_SCOPE_NONE || alpha_a_scope > MX_SCOPE_ROW || (alpha_a_scope != MX_SCOPE_NONE && !alpha_a))
        return MX_ERR_INVALID_ARG;
    if (sb2_scope != MX_SCOPE_TENSOR && sb2_scope != MX_SCOPE_ROW) return MX_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(qb) || !aligned16(sb) || !aligned16(d) || (N % 8) != 0 || (ldd % 8) != 0)
        return MX_ERR_ALIGNMENT;
    if ((K % 64) != 0 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    mxk::DqGemmArgs g{};
    g.a = static_cast<const uint16_t*>(a);
    g.alpha_a = alpha_a; g.alpha_a_scope = alpha_a ? (int)alpha_a_scope : 0;
    g.qb = qb; g.sb = sb; g.sb2 = sb2; g.sb2_scope = sb2_scope == MX_SCOPE_TENSOR ? 1 : 2;
    g.M = M; g.N = N; g.K = K; g.d = static_cast<uint16_t*>(d); g.ldd = ldd;
    return from_cuda(mxk::launch_dq_gemm(g, mxk::device_sm_count(), stream));
}

mx_status mx_wgrad_bf16_dq_nvfp4(const void* dy, const uint8_t* qx, const uint8_t* sx, const float* sx2,
                                 mx_scope sx2_scope, int64_t T, int64_t O, int64_t H, void* dw, int64_t ldd,
                                 cudaStream_t stream) {
    if (!dy || !qx || !sx || !sx2 || !dw || T <= 0 || O <= 0 || H <= 0 || ldd < H) return MX_ERR_INVALID_ARG;
    if (sx2_scope != MX_SCOPE_TENSOR && sx2_scope != MX_SCOPE_ROW) return MX_ERR_INVALID_ARG;
    if (!aligned16(dy) || !aligned16(qx) || !aligned16(sx) || !aligned16(dw) || (ldd % 8) != 0 || (O % 8) != 0)
        return MX_ERR_ALIGNMENT;
    if ((T % 64) != 0 || (H % 32) != 0 || O >= (int64_t(1) << 31) || H >= (int64_t(1) << 31) ||
        T >= (int64_t(1) << 31))
        return MX_ERR_UNSUPPORTED;
    mxk::DqGemmArgs g{};
    g.a = static_cast<const uint16_t*>(dy);
    g.alpha_a = nullptr; g.alpha_a_scope = 0;
    g.qb = qx; g.sb = sx; g.sb2 = sx2; g.sb2_scope = sx2_scope == MX_SCOPE_TENSOR ? 1 : 3;
    g.M = O; g.N = H; g.K = T; g.d = static_cast<uint16_t*>(dw); g.ldd = ldd;
    g.wgrad = true;
    return from_cuda(mxk::launch_dq_gemm(g, mxk::device_sm_count(), stream));
}

mx_status mx_fp8_blockwise_gemm(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb, int64_t M,
                                int64_t N, int64_t K, void* d, int64_t ldd, cudaStream_t stream) {
    if (!a || !sa || !b || !sb || !d || M <= 0 || N <= 0 || K <= 0 || ldd < N) return MX_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d) || (reinterpret_cast<uintptr_t>(sa) & 3) ||
        (reinterpret_cast<uintptr_t>(sb) & 3) || (N % 8) != 0 || (ldd % 8) != 0)
        return MX_ERR_ALIGNMENT;
    if ((K % 128) != 0 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    mxk::BwGemmArgs g{};
    g.a = a; g.sa = sa; g.b = b; g.sb = sb; g.M = M; g.N = N; g.K = K;
    g.d = static_cast<uint16_t*>(d); g.ldd = ldd;
    g.b_row_scales = false;
    return from_cuda(mxk::launch_fp8_blockwise_gemm(g, mxk::device_sm_count(), stream));
}

mx_status mx_fp8_blockwise_gemm_wgrad(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb, int64_t M,
                                      int64_t N, int64_t K, void* d, int64_t ldd, cudaStream_t stream) {
    if (!a || !sa || !b || !sb || !d || M <= 0 || N <= 0 || K <= 0 || ldd < N) return MX_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d) || (reinterpret_cast<uintptr_t>(sa) & 3) ||
        (reinterpret_cast<uintptr_t>(sb) & 3) || (N % 8) != 0 || (ldd % 8) != 0)
        return MX_ERR_ALIGNMENT;
    if ((K % 128) != 0 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    mxk::BwGemmArgs g{};
    g.a = a; g.sa = sa; g.b = b; g.sb = sb; g.M = M; g.N = N; g.K = K;
    g.d = static_cast<uint16_t*>(d); g.ldd = ldd;
    g.b_row_scales = true;
    return from_cuda(mxk::launch_fp8_blockwise_gemm(g, mxk::device_sm_count(), stream));
}

mx_status mx_grouped_scaled_gemm(mx_format fmt, int64_t G, const int64_t* group_offsets, int64_t total_rows,
                                 const uint8_t* a, const uint8_t* sa, const float* alpha_a_rows, const uint8_t* b,
                                 const uint8_t* sb, const float* alpha_b_groups, int64_t N, int64_t K, void* d,
                                 cudaStream_t stream) {
    mx_status st = validate_gemm_common(fmt, a, sa, b, sb, N, K, d);
    if (st != MX_OK) return st;
    if (G <= 0 || G > MX_MAX_GROUPS || !group_offsets || total_rows <= 0) return MX_ERR_INVALID_ARG;
    if (!aligned16(group_offsets)) return MX_ERR_ALIGNMENT;
    if ((N % 8) != 0) return MX_ERR_ALIGNMENT;
    mxk::GemmArgs g{};
    g.fmt = fmt == MX_FMT_MXFP8 ? 0 : 1;
    g.a = a; g.sa = sa; g.alpha_a = alpha_a_rows; g.alpha_a_scope = alpha_a_rows ? 2 : 0;
    g.b = b; g.sb = sb; g.alpha_b = alpha_b_groups; g.alpha_b_scope = alpha_b_groups ? 2 : 0;
    g.M = total_rows; g.N = N; g.K = K; g.d = static_cast<uint16_t*>(d); g.ldd = N;
    g.G = G; g.group_offsets = group_offsets;
    return from_cuda(mxk::launch_scaled_gemm(g, mxk::device_sm_count(), stream));
}

mx_status mx_count_mismatch(const uint8_t* x, const uint8_t* y, int64_t nbytes, unsigned long long* count,
                            cudaStream_t stream) {
    if (!x || !y || !count || nbytes < 0) return MX_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return MX_ERR_ALIGNMENT;
    if (nbytes == 0) return MX_OK;
    return from_cuda(mxk::launch_mismatch(x, y, nbytes, count, mxk::device_sm_count(), stream));
}

mx_status mx_check_device_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return MX_ERR_CUDA;
    const uint32_t a = mxk::read_and_clear_device_status(), b = mxk::read_and_clear_mxfp8_status();
    if (a == 0xFFFFFFFFu || b == 0xFFFFFFFFu) return MX_ERR_CUDA;
    return (a | b) ? MX_ERR_TIMEOUT : MX_OK;
}

mx_status mx_check_stream_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MX_ERR_CUDA;
    const uint32_t a = mxk::read_and_clear_device_status_on(stream), b = mxk::read_and_clear_mxfp8_status_on(stream);
    if (a == 0xFFFFFFFFu || b == 0xFFFFFFFFu) return MX_ERR_CUDA;
    return (a | b) ? MX_ERR_TIMEOUT : MX_OK;
}

mx_status mx_watchdog_selftest(mx_watchdog_unit unit, uint64_t limit_ns, cudaStream_t stream) {
    if (limit_ns < 1000u || limit_ns > 1000000000u) return MX_ERR_INVALID_ARG;
    if (unit == MX_WATCHDOG_GEMM) return from_cuda(mxk::launch_watchdog_selftest(limit_ns, stream));
    if (unit == MX_WATCHDOG_MXFP8) return from_cuda(mxk::launch_mxfp8_watchdog_selftest(limit_ns, stream));
    return MX_ERR_INVALID_ARG;
}

}  // extern "C"
