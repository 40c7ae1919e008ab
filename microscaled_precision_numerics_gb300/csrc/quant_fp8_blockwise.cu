// quant_fp8_blockwise.cu -- blockwise FP8 (E4M3) quantizers: [1, 128] tiles of activations and
// gradients, [128, 128] blocks of weights, one scale per tile or block.
//
// Source: NVIDIA NeMo RL FP8 page, section "FP8 nas camadas lineares" (E4M3 values; weights in
// [128, 128] blocks, input activations and output gradients in [1, 128] tiles, an FP32 scale per
// block, the recipe of the DeepSeek-V3 report) and section "Opções avançadas" (power-of-two scales
// instead of FP32).  Per block, with amax = max |x|:
//   FP32 scale      s = fp32(amax / 448), code = E4M3_rne_satfinite(fp32(x / s)); amax = 0 gives
//                   s = 0 and the code of x * 0 (a signed zero)
//   power of two    k = the smallest integer with 448 * 2^k >= amax, clamped to [-127, 127]
//                   (amax = 0 gives -127); s = 2^k; code = E4M3_rne_satfinite(x * 2^-k), the
//                   scaling exact.  k + 127 is an E8M0 byte: written four times per block row into
//                   the MXFP8 GEMM scale layout (one byte per 32 elements), so the MXFP8 tensor-core
//                   GEMM consumes power-of-two blockwise operands unchanged.
//
// Two kernels, both bound by HBM:
//   fp8bw_rowwise_kernel   [1, 128] tiles along a row: 16 lanes per tile, 16-byte loads, four tile
//                          pairs in flight per warp, a grid of resident CTAs striding over tile pairs.
//   fp8bw_tile_kernel      one 128 x 128 BF16 tile per CTA (256 threads, 8 rows x 8 columns each):
//                          WEIGHT mode -- one [128, 128] block: row-major codes, the same codes
//                          transposed, one scale; ACT mode -- [1, 128] tiles along rows and/or along
//                          columns (the column-wise copy stored transposed) from one read of x.
//                          Transposed codes go through an 8 x 8 byte transpose in registers and a
//                          swizzled 16 KB shared-memory tile, so both outputs leave in full 128-byte rows.

#include <cstdint>
#include <cuda_runtime.h>

#include "mx_internal.h"

namespace mxk {
namespace {

constexpr float E4M3_MAX = 448.0f;

// Power-of-two exponent of one block from its amax (FP32 bits of a non-negative BF16 value):
// amax = 1.m * 2^(E-127) gives 448 * 2^(E-135) = 1.75 * 2^(E-127), enough iff 1.m <= 1.75; one more
// otherwise.  448 * 2^(E-136) = 0.875 * 2^(E-127) < amax, so nothing smaller fits.
__device__ __forceinline__ int pow2_exponent(uint32_t amax_bits) {
    const uint32_t E = amax_bits >> 23, mant = amax_bits & 0x7FFFFFu;
    if (E == 0) return -127;                  // zero or FP32-subnormal amax: below 448 * 2^-127
    int k = (int)E - 135 + (mant > 0x600000u ? 1 : 0);
    return k < -127 ? -127 : (k > 127 ? 127 : k);
}

// 2^-k as FP32 (k in [-127, 126]: a normal number).
__device__ __forceinline__ float pow2_neg(int k) { return __uint_as_float((uint32_t)(127 - k) << 23); }

// The scale applied per element: multiply by `mul` (power of two) or divide by `div` (FP32 scale).
struct BlockScale {
    float mul;       // power of two: 2^-k; FP32: unused
    float div;       // FP32: s (0 for an all-zero block); power of two: unused
    float s;         // the stored FP32 scale
    uint32_t e8;     // power of two: k + 127
};

template <bool POW2>
__device__ __forceinline__ BlockScale block_scale(uint32_t amax_bf16) {
    BlockScale b;
    const uint32_t bits = amax_bf16 << 16;
    if constexpr (POW2) {
        const int k = pow2_exponent(bits);
        b.mul = pow2_neg(k);
        b.div = 0.0f;
        b.s = __uint_as_float((uint32_t)(k + 127) << 23);
        if (k == -127) b.s = __uint_as_float(0x00400000u);   // 2^-127 (FP32 subnormal)
        b.e8 = (uint32_t)(k + 127);
    } else {
        b.s = __fdiv_rn(__uint_as_float(bits), E4M3_MAX);
        b.div = b.s;
        b.mul = 0.0f;
        b.e8 = 0;
    }
    return b;
}

template <bool POW2>
__device__ __forceinline__ float scaled(float x, const BlockScale& b) {
    if constexpr (POW2) {
        return x * b.mul;
    } else {
        return b.div == 0.0f ? x * 0.0f : __fdiv_rn(x, b.div);
    }
}

// Eight BF16 (one 16-byte chunk) -> eight E4M3 codes (two words, element 0 in the low byte).
template <bool POW2>
__device__ __forceinline__ uint2 quant8(const uint4& v, const BlockScale& b) {
    uint2 r;
    r.x = cvt_e4m3x4(scaled<POW2>(bf16_lo(v.x), b), scaled<POW2>(bf16_hi(v.x), b), scaled<POW2>(bf16_lo(v.y), b),
                     scaled<POW2>(bf16_hi(v.y), b));
    r.y = cvt_e4m3x4(scaled<POW2>(bf16_lo(v.z), b), scaled<POW2>(bf16_hi(v.z), b), scaled<POW2>(bf16_lo(v.w), b),
                     scaled<POW2>(bf16_hi(v.w), b));
    return r;
}

__device__ __forceinline__ uint32_t chunk_absmax(const uint4& v) {
    uint32_t m = absmax_bf16x2(0u, v.x);
    m = absmax_bf16x2(m, v.y);
    m = absmax_bf16x2(m, v.z);
    m = absmax_bf16x2(m, v.w);
    return fold_halves(m);
}

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// ---------------------------------------------------------------------------------------------
// [1, 128] tiles along rows.  Tile t = r * (K / 128) + b; a warp takes pairs of consecutive tiles
// (lanes 0..15 the even one, 16..31 the odd one), RW_U pairs per pass.
// ---------------------------------------------------------------------------------------------
constexpr int RW_THREADS = 256;
constexpr int RW_U = 4;
constexpr int RW_CTAS_PER_SM = 4;

template <bool POW2>
__global__ void __launch_bounds__(RW_THREADS, RW_CTAS_PER_SM)
fp8bw_rowwise_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t K, int64_t ldx, uint8_t* __restrict__ q,
                     float* __restrict__ s, uint8_t* __restrict__ sf) {
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, c = lane & 15;
    const int64_t nb = K >> 7, T = R * nb, pairs = (T + 1) >> 1;
    const int64_t nct = nb;                        // 4-column tiles of the E8M0 layout per row band
    const int64_t warp = (int64_t)blockIdx.x * (RW_THREADS / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (RW_THREADS / 32);
    for (int64_t p0 = warp * RW_U; p0 < pairs; p0 += nwarps * RW_U) {
        uint4 v[RW_U];
        int64_t r[RW_U], b[RW_U];
#pragma unroll
        for (int u = 0; u < RW_U; ++u) {
            const int64_t t = 2 * (p0 + u) + half;
            r[u] = t / nb;
            b[u] = t - r[u] * nb;
            v[u] = t < T ? ldg16(x + r[u] * ldx + b[u] * 128 + c * 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < RW_U; ++u) {
            uint32_t m = chunk_absmax(v[u]);
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            if (r[u] >= R) continue;
            const BlockScale bs = block_scale<POW2>(m);
            const uint2 codes = quant8<POW2>(v[u], bs);
            *reinterpret_cast<uint2*>(q + r[u] * K + b[u] * 128 + c * 8) = codes;
            if (c == 0) {
                s[r[u] * nb + b[u]] = bs.s;
                if (POW2 && sf)
                    *reinterpret_cast<uint32_t*>(sf + sf_offset(r[u], 4 * b[u], nct)) = bs.e8 * 0x01010101u;
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// 128 x 128 tiles.  Thread t: column chunk c = t % 16 (columns 8c..8c+7 of the tile), row group
// g = t / 16 (rows 8g..8g+7).  The transposed staging tile holds, for tile column j, 128 code bytes
// (one per tile row) in 16 units of 8 bytes; unit g of column j sits at unit position g ^ (j / 8 % 16),
// so a half-warp's 8-byte stores (16 different column chunks) and a quarter-warp's 16-byte loads
// (one column's 128 bytes) are free of bank conflicts.
// ---------------------------------------------------------------------------------------------
constexpr int TL_THREADS = 256;
constexpr int TL_CTAS_PER_SM = 3;
enum { MODE_WEIGHT = 0, MODE_ACT = 1 };

struct TileArgs {
    const uint16_t* x; int64_t R, C, ldx, x_batch;      // x [G][R, ldx]; batch stride in elements
    // WEIGHT: q_row [G][R, C], q_col [G][C, R], s_blk [G][ceil(R/128), ceil(C/128)],
    //         sf_row [G][scale bytes (R, C)], sf_col [G][scale bytes (C, R)].
    // ACT:    q_row [R, C] with s_row [R, C/128] and sf_row; q_col [C, R] with s_col [C, R/128] and sf_col.
    uint8_t* q_row; uint8_t* q_col;
    float* s_blk; float* s_row; float* s_col;
    uint8_t* sf_row; uint8_t* sf_col;
    int64_t sf_row_bytes, sf_col_bytes;                 // per matrix (WEIGHT)
};

// 4 x 4 byte transpose: rows a, b, c, d (byte j = column j) -> column words (byte i = row i).
__device__ __forceinline__ void transpose4x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t out[4]) {
    const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(a, b, 0x7362);
    const uint32_t t2 = __byte_perm(c, d, 0x5140), t3 = __byte_perm(c, d, 0x7362);
    out[0] = __byte_perm(t0, t2, 0x5410);
    out[1] = __byte_perm(t0, t2, 0x7632);
    out[2] = __byte_perm(t1, t3, 0x5410);
    out[3] = __byte_perm(t1, t3, 0x7632);
}

// Writes the thread's 8 x 8 codes (cw[i] = row i, columns 0..7) transposed into the staging tile.
__device__ __forceinline__ void stage_transposed(uint8_t* st, const uint2 cw[8], int c, int g) {
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t w0 = h ? cw[0].y : cw[0].x, w1 = h ? cw[1].y : cw[1].x, w2 = h ? cw[2].y : cw[2].x,
                       w3 = h ? cw[3].y : cw[3].x, w4 = h ? cw[4].y : cw[4].x, w5 = h ? cw[5].y : cw[5].x,
                       w6 = h ? cw[6].y : cw[6].x, w7 = h ? cw[7].y : cw[7].x;
        transpose4x4(w0, w1, w2, w3, lo);
        transpose4x4(w4, w5, w6, w7, hi);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = 8 * c + 4 * h + j;
            *reinterpret_cast<uint2*>(st + col * 128 + ((g ^ c) << 3)) = make_uint2(lo[j], hi[j]);
        }
    }
}

// Stores the staged transposed codes: tile column j -> output row (c0 + j), bytes r0 .. r0 + 127.
__device__ __forceinline__ void store_transposed(const uint8_t* st, uint8_t* out, int64_t ld, int64_t r0,
                                                 int64_t c0, int64_t R, int64_t C) {
    const int p = threadIdx.x & 7;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int j = (threadIdx.x >> 3) + 32 * k;
        const int f = (j >> 3) & 15;
        uint4 w = *reinterpret_cast<const uint4*>(st + j * 128 + (((2 * p) ^ (f & 14)) << 3));
        if (f & 1) w = make_uint4(w.z, w.w, w.x, w.y);
        if (c0 + j < C && r0 + 16 * p < R)
            *reinterpret_cast<uint4*>(out + (c0 + j) * ld + r0 + 16 * p) = w;
    }
}

template <int MODE, bool POW2, bool ROW, bool COL>
__global__ void __launch_bounds__(TL_THREADS, (ROW && COL) ? 2 : TL_CTAS_PER_SM) fp8bw_tile_kernel(const TileArgs a) {
    __shared__ __align__(16) uint8_t st[128 * 128];
    __shared__ uint32_t red[8][16][4];
    __shared__ uint32_t red_all[8];

    const int t = threadIdx.x, c = t & 15, g = t >> 4, warp = t >> 5;
    const int64_t bz = blockIdx.z;
    const int64_t r0 = (int64_t)blockIdx.y * 128, c0 = (int64_t)blockIdx.x * 128;
    const int64_t R = a.R, C = a.C;
    const uint16_t* x = a.x + bz * a.x_batch;
    const bool col_ok = c0 + 8 * c < C;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = r0 + 8 * g + i;
        v[i] = (col_ok && r < R) ? ldg16(x + r * a.ldx + c0 + 8 * c) : make_uint4(0, 0, 0, 0);
    }

    uint2 cw[8];
    if constexpr (MODE == MODE_WEIGHT) {
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = max(m, chunk_absmax(v[i]));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if ((t & 31) == 0) red_all[warp] = m;
        __syncthreads();
        m = red_all[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) m = max(m, red_all[w]);
        const BlockScale bs = block_scale<POW2>(m);
#pragma unroll
        for (int i = 0; i < 8; ++i) cw[i] = quant8<POW2>(v[i], bs);

        const int64_t tr = gridDim.y, tc = gridDim.x;
        uint8_t* q_row = a.q_row + bz * R * C;
        uint8_t* q_col = a.q_col + bz * R * C;
        if (col_ok) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t r = r0 + 8 * g + i;
                if (r < R) *reinterpret_cast<uint2*>(q_row + r * C + c0 + 8 * c) = cw[i];
            }
        }
        if (t == 0) a.s_blk[(bz * tr + blockIdx.y) * tc + blockIdx.x] = bs.s;
        if (POW2) {
            const uint32_t word = bs.e8 * 0x01010101u;
            if (a.sf_row && t < 128 && r0 + t < R)
                *reinterpret_cast<uint32_t*>(a.sf_row + bz * a.sf_row_bytes +
                                             sf_offset(r0 + t, 4 * (int64_t)blockIdx.x, sf_col_tiles(C, 32))) = word;
            if (a.sf_col && t >= 128 && c0 + (t - 128) < C)
                *reinterpret_cast<uint32_t*>(a.sf_col + bz * a.sf_col_bytes +
                                             sf_offset(c0 + (t - 128), 4 * (int64_t)blockIdx.y, sf_col_tiles(R, 32))) =
                    word;
        }
        stage_transposed(st, cw, c, g);
        __syncthreads();
        store_transposed(st, q_col, R, r0, c0, R, C);
    } else {
        if constexpr (ROW) {
            // [1, 128] tiles along the row: the 16 lanes of a half-warp hold one row's 128 values.
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t m = chunk_absmax(v[i]);
#pragma unroll
                for (int o = 8; o >= 1; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                const BlockScale bs = block_scale<POW2>(m);
                const uint2 codes = quant8<POW2>(v[i], bs);
                const int64_t r = r0 + 8 * g + i;
                *reinterpret_cast<uint2*>(a.q_row + r * C + c0 + 8 * c) = codes;
                if (c == 0) {
                    a.s_row[r * (C >> 7) + blockIdx.x] = bs.s;
                    if (POW2 && a.sf_row)
                        *reinterpret_cast<uint32_t*>(a.sf_row + sf_offset(r, 4 * (int64_t)blockIdx.x, C >> 7)) =
                            bs.e8 * 0x01010101u;
                }
            }
        }
        if constexpr (COL) {
            // [1, 128] tiles along the column (128 rows of one column): per-column maxima of the
            // thread's 8 rows, then over the 16 row groups (lane pair, then the 8 warps).
            uint32_t cm[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t m = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t w = j == 0 ? v[i].x : j == 1 ? v[i].y : j == 2 ? v[i].z : v[i].w;
                    m = absmax_bf16x2(m, w);
                }
                m = __vmaxu2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
                cm[j] = m;
            }
            if ((t & 31) < 16) {
#pragma unroll
                for (int j = 0; j < 4; ++j) red[warp][c][j] = cm[j];
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t m = red[0][c][j];
#pragma unroll
                for (int w = 1; w < 8; ++w) m = __vmaxu2(m, red[w][c][j]);
                cm[j] = m;
            }
            BlockScale bs[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) bs[j] = block_scale<POW2>(j & 1 ? cm[j >> 1] >> 16 : cm[j >> 1] & 0xFFFFu);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint4 w = v[i];
                cw[i].x = cvt_e4m3x4(scaled<POW2>(bf16_lo(w.x), bs[0]), scaled<POW2>(bf16_hi(w.x), bs[1]),
                                     scaled<POW2>(bf16_lo(w.y), bs[2]), scaled<POW2>(bf16_hi(w.y), bs[3]));
                cw[i].y = cvt_e4m3x4(scaled<POW2>(bf16_lo(w.z), bs[4]), scaled<POW2>(bf16_hi(w.z), bs[5]),
                                     scaled<POW2>(bf16_lo(w.w), bs[6]), scaled<POW2>(bf16_hi(w.w), bs[7]));
            }
            if (g == 0 && col_ok) {
                const int64_t nbr = R >> 7;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int64_t col = c0 + 8 * c + j;
                    a.s_col[col * nbr + blockIdx.y] = bs[j].s;
                    if (POW2 && a.sf_col)
                        *reinterpret_cast<uint32_t*>(a.sf_col + sf_offset(col, 4 * (int64_t)blockIdx.y, nbr)) =
                            bs[j].e8 * 0x01010101u;
                }
            }
            stage_transposed(st, cw, c, g);
            __syncthreads();
            store_transposed(st, a.q_col, R, r0, c0, R, C);
        }
    }
}

template <int MODE, bool POW2, bool ROW, bool COL>
cudaError_t launch_tile(const TileArgs& a, int64_t G, cudaStream_t stream) {
    const dim3 grid((unsigned)((a.C + 127) / 128), (unsigned)((a.R + 127) / 128), (unsigned)G);
    fp8bw_tile_kernel<MODE, POW2, ROW, COL><<<grid, TL_THREADS, 0, stream>>>(a);
    return cudaGetLastError();
}

template <bool POW2>
cudaError_t launch_rowwise(const uint16_t* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q, float* s, uint8_t* sf,
                           int num_sms, cudaStream_t stream) {
    const int64_t pairs = (R * (K >> 7) + 1) >> 1;
    const int64_t warps = (pairs + RW_U - 1) / RW_U;
    const int64_t need = (warps + RW_THREADS / 32 - 1) / (RW_THREADS / 32);
    const int64_t resident = (int64_t)num_sms * RW_CTAS_PER_SM;
    const unsigned grid = (unsigned)(need < resident ? need : resident);
    fp8bw_rowwise_kernel<POW2><<<grid, RW_THREADS, 0, stream>>>(x, R, K, ldx, q, s, sf);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_blockwise_1x128(const uint16_t* x, int64_t R, int64_t K, int64_t ldx, bool pow2,
                                       uint8_t* q_row, float* s_row, uint8_t* sf_row, uint8_t* q_col, float* s_col,
                                       uint8_t* sf_col, int num_sms, cudaStream_t stream) {
    if (!q_col) {
        return pow2 ? launch_rowwise<true>(x, R, K, ldx, q_row, s_row, sf_row, num_sms, stream)
                    : launch_rowwise<false>(x, R, K, ldx, q_row, s_row, sf_row, num_sms, stream);
    }
    TileArgs a{};
    a.x = x; a.R = R; a.C = K; a.ldx = ldx; a.x_batch = 0;
    a.q_row = q_row; a.s_row = s_row; a.sf_row = sf_row;
    a.q_col = q_col; a.s_col = s_col; a.sf_col = sf_col;
    if (q_row) {
        return pow2 ? launch_tile<MODE_ACT, true, true, true>(a, 1, stream)
                    : launch_tile<MODE_ACT, false, true, true>(a, 1, stream);
    }
    return pow2 ? launch_tile<MODE_ACT, true, false, true>(a, 1, stream)
                : launch_tile<MODE_ACT, false, false, true>(a, 1, stream);
}

cudaError_t launch_fp8_blockwise_128x128(const uint16_t* w, int64_t G, int64_t O, int64_t H, bool pow2,
                                         uint8_t* q_row, uint8_t* q_col, float* s, uint8_t* sf_row, uint8_t* sf_col,
                                         cudaStream_t stream) {
    TileArgs a{};
    a.x = w; a.R = O; a.C = H; a.ldx = H; a.x_batch = O * H;
    a.q_row = q_row; a.q_col = q_col; a.s_blk = s;
    a.sf_row = sf_row; a.sf_col = sf_col;
    a.sf_row_bytes = host_scale_bytes(O, H, 32);
    a.sf_col_bytes = host_scale_bytes(H, O, 32);
    return pow2 ? launch_tile<MODE_WEIGHT, true, false, false>(a, G, stream)
                : launch_tile<MODE_WEIGHT, false, false, false>(a, G, stream);
}

}  // namespace mxk
