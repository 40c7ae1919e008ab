// mx_device.cuh -- device helpers shared by the mxnum kernels (sm_103a).
//
// Format conversions use the documented PTX cvt instructions (round-to-nearest-even, satfinite);
// scale factors and reciprocals use the IEEE round-to-nearest intrinsics (__fdiv_rn, __frcp_rn,
// __fmul_rn) so no step is contracted or approximated.  The library is built without fast-math and
// with denormals preserved.
#pragma once

#include <cstdint>
#include <cfloat>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace mxk {

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// ---------------------------------------------------------------------------------------------
// BF16 / format conversions
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two FP32 -> packed BF16 pair (round to nearest even); `lo` lands in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four FP32 -> four E4M3 bytes (RNE, satfinite), element 0 in bits 0..7.
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a0, float a1, float a2, float a3) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r) : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
    return r;
}

// One non-negative FP32 -> E4M3 byte (RNE, satfinite).
__device__ __forceinline__ uint32_t cvt_e4m3(float a) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(a));
    return r & 0xFFu;
}

// E4M3 byte -> FP32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
    uint32_t h2;
    asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h2) : "r"(code & 0xFFu));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Eight FP32 -> eight E2M1 nibbles packed in 32 bits (RNE, satfinite), element 0 in bits 0..3.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float v[8]) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// Two packed E2M1 codes (one byte) -> two FP16 values (exact); element 0 from the low nibble.
// Value of a 4-bit E2M1 code (s ee m, bias 1; e = 0 subnormal m * 0.5) from its field definition.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    const uint32_t mag = e ? (((e + 126u) << 23) | (m << 22)) : (m ? 0x3F000000u : 0u);
    return __uint_as_float(mag | ((c & 8u) << 28));
}

__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{\n\t.reg .b8 c;\n\tcvt.u8.u32 c, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, c;\n\t}" : "=r"(r) : "r"(byte & 0xFFu));
    return r;
}

// ---------------------------------------------------------------------------------------------
// Stochastic rounding onto the E2M1 grid {0, .5, 1, 1.5, 2, 3, 4, 6} with 16 random bits.
// a = |v|; a >= 6 -> 6; else lo/hi are the neighbouring grid points, f = (a - lo) / (hi - lo)
// (exact), and the result rounds up iff f > bits * 2^-16.  Returns the 4-bit code (sign kept).
// Evaluated on the FP32 bit fields (same decisions as the quotient form).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e2m1_sr(float v, uint32_t bits16) {
    // For a in [1, 6) the two grid points of each binade [2^e, 2^(e+1)) are 2^e and 1.5 * 2^e: the top
    // mantissa bit picks the lower one and f is the remaining 22 mantissa bits over 2^22, so f > bits16 *
    // 2^-16 exactly when adding 2^22 - 1 - (bits16 << 6) to the FP32 bits carries into that top bit; the
    // code 2 + 2e + m is then read off the sum (a carry out of the binade lands on the next grid point,
    // and anything from 6 up clamps to 7).  In [0.5, 1) the grid points are 0.5 and 1 and f is the whole
    // 23-bit mantissa over 2^23: the same carry test one bit up.  Below 0.5 (grid 0 and 0.5) f = 2a, and
    // 2a > bits16 * 2^-16 is compared as a * 2^17 > bits16 in FP32 (both sides exact).
    const uint32_t u = __float_as_uint(v) & 0x7FFFFFFFu;
    const uint32_t c_norm = min(((u + (0x3FFFFFu - (bits16 << 6))) >> 22) - 252u, 7u);
    const uint32_t c_half = ((u + (0x7FFFFFu - (bits16 << 7))) >> 23) - 125u;
    const float fbits = __fsub_rn(__uint_as_float(0x4B000000u | bits16), 8388608.0f);   // bits16 as FP32, exactly
    const uint32_t c_small = __fmul_rn(__uint_as_float(u), 131072.0f) > fbits ? 1u : 0u;
    const uint32_t code = u >= 0x3F800000u ? c_norm : (u >= 0x3F000000u ? c_half : c_small);
    return code | ((__float_as_uint(v) >> 28) & 8u);
}

// ---------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11): counter (c0..c3), key (k0, k1).
// ---------------------------------------------------------------------------------------------
struct U4 { uint32_t x, y, z, w; };

__device__ __forceinline__ U4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                            uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int rnd = 0; rnd < 10; ++rnd) {
        // one widening multiply gives both halves of each 64-bit product
        const unsigned long long p0 = (unsigned long long)0xD2511F53u * c0;
        const unsigned long long p1 = (unsigned long long)0xCD9E8D57u * c2;
        const uint32_t lo0 = (uint32_t)p0, hi0 = (uint32_t)(p0 >> 32);
        const uint32_t lo1 = (uint32_t)p1, hi1 = (uint32_t)(p1 >> 32);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += 0x9E3779B9u; k1 += 0xBB67AE85u;
    }
    return U4{c0, c1, c2, c3};
}

// RHT sign mask: bit j set means d_j = -1.
__device__ __forceinline__ uint32_t rht_sign_mask(uint64_t seed) {
    return philox4x32_10(0u, 0u, 1u, 0u, (uint32_t)seed, (uint32_t)(seed >> 32)).x & 0xFFFFu;
}

// In-register 16-point transform without the final 1/4: signs, then butterflies with strides 1, 2, 4, 8.
__device__ __forceinline__ void rht16_unscaled(float v[16], uint32_t signmask) {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = ((signmask >> j) & 1u) ? -v[j] : v[j];
#pragma unroll
    for (int h = 1; h < 16; h *= 2) {
#pragma unroll
        for (int i = 0; i < 16; i += 2 * h) {
#pragma unroll
            for (int j = i; j < i + h; ++j) {
                const float a = v[j], b = v[j + h];
                v[j] = __fadd_rn(a, b);
                v[j + h] = __fsub_rn(a, b);
            }
        }
    }
}

// In-register 16-point transform: signs, butterflies with strides 1, 2, 4, 8, then x 1/4.
__device__ __forceinline__ void rht16_inplace(float v[16], uint32_t signmask) {
    rht16_unscaled(v, signmask);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], 0.25f);
}

// ---------------------------------------------------------------------------------------------
// NVFP4 block-scale arithmetic (FP32, round to nearest, in the documented order).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float nvfp4_second_scale(float amax) { return __fdiv_rn(amax, 2688.0f); }

// bs = E4M3(fp32(fp32(amax_b / m) / S)) with m = 6 (the block maximum maps to the E2M1 maximum) or,
// for the Four-over-Six alternative, m = 4.
__device__ __forceinline__ uint32_t nvfp4_block_scale_m(float amax_b, float S, float m) {
    if (S == 0.0f) return 0u;
    return cvt_e4m3(__fdiv_rn(__fdiv_rn(amax_b, m), S));
}
__device__ __forceinline__ uint32_t nvfp4_block_scale(float amax_b, float S) { return nvfp4_block_scale_m(amax_b, S, 6.0f); }

__device__ __forceinline__ float nvfp4_block_recip(uint32_t bs, float S) {
    const float d = __fmul_rn(e4m3_to_f32(bs), S);
    if (d == 0.0f) return 0.0f;
    return fminf(__frcp_rn(d), FLT_MAX);
}

// ---------------------------------------------------------------------------------------------
// GEMM scale layout: 512-byte tiles of 128 rows x 4 scale columns, tile-row-major; inside a tile
// (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4).  `nct` = number of 4-column tiles per row band.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t nct) {
    return (((r >> 7) * nct + (c >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (c & 3);
}

__host__ __device__ __forceinline__ int64_t sf_col_tiles(int64_t k, int block) {
    return (k / block + 3) / 4;
}

// Max of |bf16| over the two halves of each word, as 16-bit integers (NaN-free inputs).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) {
    return __vmaxu2(acc, w & 0x7FFF7FFFu);
}
__device__ __forceinline__ uint32_t fold_halves(uint32_t m2) { return max(m2 & 0xFFFFu, m2 >> 16); }

// ---------------------------------------------------------------------------------------------
// Expert-group tables for the grouped scale layout: group g's rows [off[g], off[g+1]) start at
// padded 128-row tile ptile[g] = sum over j < g of ceil(m_j / 128).  Built by a whole block:
// offsets copied to shared memory, tile counts scanned in parallel (warp shuffles + one pass over
// the warp totals).  s_off needs G + 1 entries, s_ptile G + 1 entries, s_warp 32 entries.
// ---------------------------------------------------------------------------------------------
// Tile prefix only, reading the offsets through `off` (shared or global memory).
template <int ROWS = 128>
__device__ __forceinline__ void scan_group_tiles(const int64_t* off, int G, int* s_ptile, int* s_warp) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, wid = tid >> 5, nwarps = nthr >> 5;
    // thread tid owns groups [tid * per, tid * per + per)
    const int per = (G + nthr - 1) / nthr;
    int local = 0;
    for (int k = 0; k < per; ++k) {
        const int g = tid * per + k;
        if (g < G) local += (int)((off[g + 1] - off[g] + ROWS - 1) / ROWS);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o) w += v;
        }
        if (lane < nwarps) s_warp[lane] = w;   // inclusive warp totals
    }
    __syncthreads();
    int run = incl - local + (wid > 0 ? s_warp[wid - 1] : 0);   // exclusive prefix of this thread's first group
    for (int k = 0; k < per; ++k) {
        const int g = tid * per + k;
        if (g < G) {
            s_ptile[g] = run;
            run += (int)((off[g + 1] - off[g] + ROWS - 1) / ROWS);
        }
        if (g == G - 1) s_ptile[G] = run;
    }
    __syncthreads();
}

__device__ __forceinline__ void load_group_tables(const int64_t* __restrict__ offsets, int G, int64_t* s_off,
                                                  int* s_ptile, int* s_warp) {
    for (int i = threadIdx.x; i <= G; i += blockDim.x) s_off[i] = __ldg(offsets + i);
    __syncthreads();
    scan_group_tiles(s_off, G, s_ptile, s_warp);
}

// Group of row r: the g with s_off[g] <= r < s_off[g + 1] (empty groups are skipped).
__device__ __forceinline__ int find_group(const int64_t* s_off, int G, int64_t r) {
    int lo = 0, hi = G;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= r) lo = mid; else hi = mid;
    }
    return lo;
}

// Row of r in the grouped scale layout.
__device__ __forceinline__ int64_t grouped_scale_row(const int64_t* s_off, const int* s_ptile, int G, int64_t r) {
    const int g = find_group(s_off, G, r);
    return (int64_t)s_ptile[g] * 128 + (r - s_off[g]);
}

}  // namespace mxk

