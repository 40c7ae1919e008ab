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
// Two kernels, both meant to run at the HBM roofline; the arithmetic per element is kept small:
// block maxima on packed BF16 pairs (max of magnitudes, one instruction per pair), each BF16 value
// widened once, one scale per block computed once per lane group.
//   fp8bw_rowwise_kernel   [1, 128] tiles along a row: 4 lanes per tile (32 values each, four
//                          16-byte loads), 8 tiles per warp and pass, RW_U passes in flight; a grid
//                          of resident CTAs strides over the tiles.
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

// One block's scale: `f` is what each value is multiplied by (power of two: 2^-k) or divided by
// (FP32: s, 0 for an all-zero block); `s` the stored FP32 scale; `e8` = k + 127 (power of two).
struct BlockScale {
    float f;
    float s;
    uint32_t e8;
};

template <bool POW2>
__device__ __forceinline__ BlockScale block_scale(uint32_t amax_bf16) {
    BlockScale b;
    const uint32_t bits = amax_bf16 << 16;
    if constexpr (POW2) {
        const int k = pow2_exponent(bits);
        b.f = __uint_as_float((uint32_t)(127 - k) << 23);            // 2^-k, k <= 126 for finite BF16
        b.s = k == -127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(k + 127) << 23);
        b.e8 = (uint32_t)(k + 127);
    } else {
        b.s = __fdiv_rn(__uint_as_float(bits), E4M3_MAX);
        b.f = b.s;
        b.e8 = 0;
    }
    return b;
}

template <bool POW2>
__device__ __forceinline__ float scaled(float x, float f) {
    if constexpr (POW2) {
        return x * f;
    } else {
        return f == 0.0f ? x * 0.0f : __fdiv_rn(x, f);
    }
}

// max(|a|, |b|) of each BF16 half of two packed pairs; the sign bits of the result are meaningless
// (masked once at the end of a reduction).  Inputs hold no NaN.
__device__ __forceinline__ uint32_t max_abs2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Largest magnitude of the two halves of a reduced pair (BF16 bits, low 16 bits).
__device__ __forceinline__ uint32_t fold_abs(uint32_t m) {
    m &= 0x7FFF7FFFu;
    return max(m & 0xFFFFu, m >> 16);
}

__device__ __forceinline__ uint32_t chunk_max_abs2(const uint4& v) {
    return max_abs2(max_abs2(v.x, v.y), max_abs2(v.z, v.w));
}

// Eight BF16 values (one 16-byte chunk) widened to FP32.
__device__ __forceinline__ void widen8(const uint4& v, float f[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Eight values, one scale -> eight E4M3 codes (element 0 in the low byte).
template <bool POW2>
__device__ __forceinline__ uint2 quant8(const float f[8], float s) {
    uint2 r;
    r.x = cvt_e4m3x4(scaled<POW2>(f[0], s), scaled<POW2>(f[1], s), scaled<POW2>(f[2], s), scaled<POW2>(f[3], s));
    r.y = cvt_e4m3x4(scaled<POW2>(f[4], s), scaled<POW2>(f[5], s), scaled<POW2>(f[6], s), scaled<POW2>(f[7], s));
    return r;
}

// Eight values, one scale per value (eight columns).
template <bool POW2>
__device__ __forceinline__ uint2 quant8_cols(const float f[8], const float s[8]) {
    uint2 r;
    r.x = cvt_e4m3x4(scaled<POW2>(f[0], s[0]), scaled<POW2>(f[1], s[1]), scaled<POW2>(f[2], s[2]),
                     scaled<POW2>(f[3], s[3]));
    r.y = cvt_e4m3x4(scaled<POW2>(f[4], s[4]), scaled<POW2>(f[5], s[5]), scaled<POW2>(f[6], s[6]),
                     scaled<POW2>(f[7], s[7]));
    return r;
}

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// ---------------------------------------------------------------------------------------------
// [1, 128] tiles along rows.  Tile t = r * (K / 128) + b.  Lane l of a warp works on tile
// (8 * pass + l / 4) with chunks (l % 4) + 4 j, j = 0..3 (8 values each): per load instruction the
// warp reads 64 contiguous bytes of each of 8 tiles.  The row of a tile comes from a multiply-shift
// division by K / 128 (exact for t < 2^31).
// ---------------------------------------------------------------------------------------------
constexpr int RW_THREADS = 256;
constexpr int RW_U = 2;
constexpr int RW_CTAS_PER_SM = 4;

// n / d = (n * m) >> (32 + l) for 0 <= n < 2^31, with l = ceil(log2 d) and m = ceil(2^(32+l) / d):
// the product overshoots n / d by less than n / 2^(32+l) < 2^-l <= 1 / d, which cannot reach the next
// integer.
struct FastDiv {
    uint64_t m;
    uint32_t shift;
};

FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const unsigned __int128 num = (unsigned __int128)1 << (32 + l);
    return FastDiv{(uint64_t)((num + d - 1) / d), 32 + l};
}

__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
    return (uint32_t)(((uint64_t)n * f.m) >> f.shift);
}

template <bool POW2>
__global__ void __launch_bounds__(RW_THREADS, RW_CTAS_PER_SM)
fp8bw_rowwise_kernel(const uint16_t* __restrict__ x, uint32_t R, uint32_t nb, int64_t ldx, uint8_t* __restrict__ q,
                     float* __restrict__ s, uint8_t* __restrict__ sf, FastDiv div_nb) {
    const int lane = threadIdx.x & 31;
    const int sub = lane & 3;
    const uint32_t T = R * nb;
    const uint32_t warp = blockIdx.x * (RW_THREADS / 32) + (threadIdx.x >> 5);
    const uint32_t nwarps = gridDim.x * (RW_THREADS / 32);
    for (uint32_t t0 = warp * (8 * RW_U); t0 < T; t0 += nwarps * (8 * RW_U)) {
        uint4 v[RW_U][4];
        uint32_t tt[RW_U], rr[RW_U];
#pragma unroll
        for (int u = 0; u < RW_U; ++u) {
            const uint32_t t = t0 + 8 * u + (lane >> 2);
            tt[u] = t;
            const uint32_t r = fast_div(t, div_nb);
            rr[u] = r;
            const uint16_t* src = x + (int64_t)r * ldx + (t - r * nb) * 128 + sub * 8;
#pragma unroll
            for (int j = 0; j < 4; ++j) v[u][j] = t < T ? ldg16(src + 32 * j) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < RW_U; ++u) {
            uint32_t m = max_abs2(chunk_max_abs2(v[u][0]), chunk_max_abs2(v[u][1]));
            m = max_abs2(m, max_abs2(chunk_max_abs2(v[u][2]), chunk_max_abs2(v[u][3])));
            m = max_abs2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max_abs2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            const uint32_t t = tt[u];
            if (t >= T) continue;
            const BlockScale bs = block_scale<POW2>(fold_abs(m));
            uint8_t* dst = q + (int64_t)t * 128 + sub * 8;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float f[8];
                widen8(v[u][j], f);
                *reinterpret_cast<uint2*>(dst + 32 * j) = quant8<POW2>(f, bs.f);
            }
            if (sub == 0) {
                s[t] = bs.s;
                if (POW2 && sf)
                    *reinterpret_cast<uint32_t*>(sf + sf_offset(rr[u], 4 * (t - rr[u] * nb), nb)) = bs.e8 * 0x01010101u;
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// 128 x 128 tiles.  Thread t: column chunk c = t % 16 (columns 8c..8c+7 of the tile), row group
// g = t / 16 (rows 8g..8g+7); a half-warp holds 8 whole rows.  The transposed staging tile holds,
// for tile column j, 128 code bytes (one per tile row) in 16 units of 8 bytes; unit g of column j
// sits at unit position g ^ (j / 8 % 16), so a half-warp's 8-byte stores (16 different column
// chunks) and a quarter-warp's 16-byte loads (one column's 128 bytes) are free of bank conflicts.
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

// Row maxima of the 8 rows a half-warp holds (a[i] = this lane's packed pair maximum of row i):
// a butterfly that halves the rows kept at each step, so lane c of the half-warp ends with the
// maximum of row c / 2 (8 shuffles instead of 32).
__device__ __forceinline__ uint32_t half_warp_row_max(const uint32_t a[8], int c) {
    uint32_t b[4], d[2];
    const bool h8 = c & 8, h4 = c & 4, h2 = c & 2;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t send = h8 ? a[k] : a[k + 4], keep = h8 ? a[k + 4] : a[k];
        b[k] = max_abs2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 8));
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t send = h4 ? b[k] : b[k + 2], keep = h4 ? b[k + 2] : b[k];
        d[k] = max_abs2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 4));
    }
    const uint32_t send = h2 ? d[0] : d[1], keep = h2 ? d[1] : d[0];
    uint32_t e = max_abs2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 2));
    e = max_abs2(e, __shfl_xor_sync(0xFFFFFFFFu, e, 1));
    return fold_abs(e);
}

template <int MODE, bool POW2, bool ROW, bool COL>
__global__ void __launch_bounds__(TL_THREADS, (ROW && COL && !POW2) ? 2 : TL_CTAS_PER_SM) fp8bw_tile_kernel(const TileArgs a) {
    __shared__ __align__(16) uint8_t st[128 * 128];
    __shared__ uint32_t red[8][16][4];
    __shared__ __align__(16) float colf[128];
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
        uint32_t m = chunk_max_abs2(v[0]);
#pragma unroll
        for (int i = 1; i < 8; ++i) m = max_abs2(m, chunk_max_abs2(v[i]));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = max_abs2(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if ((t & 31) == 0) red_all[warp] = fold_abs(m);
        __syncthreads();
        uint32_t amax = red_all[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) amax = max(amax, red_all[w]);
        const BlockScale bs = block_scale<POW2>(amax);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float f[8];
            widen8(v[i], f);
            cw[i] = quant8<POW2>(f, bs.f);
        }

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
        // Row scales ([1, 128] tiles along rows): lane c of each half-warp owns row 8g + c / 2.
        float rowf[8];
        if constexpr (ROW) {
            uint32_t rm[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) rm[i] = chunk_max_abs2(v[i]);
            const BlockScale bs = block_scale<POW2>(half_warp_row_max(rm, c));
            const int64_t r = r0 + 8 * g + (c >> 1);
            if ((c & 1) == 0) {
                a.s_row[r * (C >> 7) + blockIdx.x] = bs.s;
                if (POW2 && a.sf_row)
                    *reinterpret_cast<uint32_t*>(a.sf_row + sf_offset(r, 4 * (int64_t)blockIdx.x, C >> 7)) =
                        bs.e8 * 0x01010101u;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) rowf[i] = __shfl_sync(0xFFFFFFFFu, bs.f, (t & 16) | (2 * i));
        }
        // Column scales ([1, 128] tiles along columns): packed maxima of the thread's 8 rows, then
        // over the 16 row groups (lane pair, then the 8 warps); thread j < 128 finishes column j.
        float cf[8];
        if constexpr (COL) {
            uint32_t cm[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t m = j == 0 ? v[0].x : j == 1 ? v[0].y : j == 2 ? v[0].z : v[0].w;
#pragma unroll
                for (int i = 1; i < 8; ++i)
                    m = max_abs2(m, j == 0 ? v[i].x : j == 1 ? v[i].y : j == 2 ? v[i].z : v[i].w);
                cm[j] = max_abs2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
            }
            if ((t & 31) < 16) {
#pragma unroll
                for (int j = 0; j < 4; ++j) red[warp][c][j] = cm[j];
            }
            __syncthreads();
            if (t < 128) {
                const int cc = t >> 3, word = (t & 7) >> 1;
                uint32_t m = red[0][cc][word];
#pragma unroll
                for (int w = 1; w < 8; ++w) m = max_abs2(m, red[w][cc][word]);
                m &= 0x7FFF7FFFu;
                const BlockScale bs = block_scale<POW2>((t & 1) ? (m >> 16) : (m & 0xFFFFu));
                colf[t] = bs.f;
                const int64_t col = c0 + t;
                if (col < C) {
                    const int64_t nbr = R >> 7;
                    a.s_col[col * nbr + blockIdx.y] = bs.s;
                    if (POW2 && a.sf_col)
                        *reinterpret_cast<uint32_t*>(a.sf_col + sf_offset(col, 4 * (int64_t)blockIdx.y, nbr)) =
                            bs.e8 * 0x01010101u;
                }
            }
            __syncthreads();
            const float4 f0 = *reinterpret_cast<const float4*>(colf + 8 * c);
            const float4 f1 = *reinterpret_cast<const float4*>(colf + 8 * c + 4);
            cf[0] = f0.x; cf[1] = f0.y; cf[2] = f0.z; cf[3] = f0.w;
            cf[4] = f1.x; cf[5] = f1.y; cf[6] = f1.z; cf[7] = f1.w;
        }
        // Each value widened once, quantized with its row scale and with its column scale.
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float f[8];
            widen8(v[i], f);
            if constexpr (ROW) {
                const int64_t r = r0 + 8 * g + i;
                *reinterpret_cast<uint2*>(a.q_row + r * C + c0 + 8 * c) = quant8<POW2>(f, rowf[i]);
            }
            if constexpr (COL) cw[i] = quant8_cols<POW2>(f, cf);
        }
        if constexpr (COL) {
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
    const int64_t tiles = R * (K >> 7);
    const int64_t warps = (tiles + 8 * RW_U - 1) / (8 * RW_U);
    const int64_t need = (warps + RW_THREADS / 32 - 1) / (RW_THREADS / 32);
    const int64_t resident = (int64_t)num_sms * RW_CTAS_PER_SM;
    const unsigned grid = (unsigned)(need < resident ? need : resident);
    fp8bw_rowwise_kernel<POW2><<<grid, RW_THREADS, 0, stream>>>(x, (uint32_t)R, (uint32_t)(K >> 7), ldx, q, s, sf,
                                                                 make_fastdiv((uint32_t)(K >> 7)));
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
                                         int num_sms, cudaStream_t stream) {
    (void)num_sms;
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
