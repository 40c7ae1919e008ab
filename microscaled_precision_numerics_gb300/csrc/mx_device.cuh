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
// 32 contiguous bytes written with one 256-bit streaming store when p is 32-byte aligned (a warp's
// store then covers whole lines in one instruction), two 16-byte stores otherwise.  (The matching
// 256-bit load made the per-token quantizer slower: 0.081 -> 0.101 ms on 65536 x 2048.)
__device__ __forceinline__ void stcs_32b(void* p, const uint4& a, const uint4& b) {
    if ((reinterpret_cast<uintptr_t>(p) & 31u) == 0) {
        asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                     :: "l"(p), "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                     : "memory");
    } else {
        __stcs(reinterpret_cast<uint4*>(p), a);
        __stcs(reinterpret_cast<uint4*>(p) + 1, b);
    }
}

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

// Two packed E2M1 codes (the low byte) -> two FP16 values (exact); element 0 from the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{\n\t.reg .b8 c;\n\tcvt.u8.u32 c, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, c;\n\t}" : "=r"(r) : "r"(byte & 0xFFu));
    return r;
}

// ---------------------------------------------------------------------------------------------
// Stochastic rounding onto the E2M1 grid {0, .5, 1, 1.5, 2, 3, 4, 6} with 16 random bits k.
// a = |v|; a >= 6 -> 6; else lo/hi are the neighbouring grid points, f = (a - lo) / (hi - lo)
// (exact), and the result rounds up iff f > k * 2^-16.  Returns the 4-bit code (sign kept).
//
// Evaluated on one FP32 bit pattern.  z = a * 2^-126 rounded up: for a >= 1 the product is exact and
// normal, its exponent field is e + 1 for a in [2^e, 2^(e+1)) and its top mantissa bit picks 2^e or
// 1.5 * 2^e, so bits(z) >> 22 = 2 + 2e + m is the code of lo, and the low 22 bits are f * 2^22.  For
// a < 1 the product is subnormal, bits(z) = ceil(a * 2^23): bits >> 22 = floor(2a) is again the code of
// lo (grid step 0.5) and the low 22 bits are ceil(f * 2^22).  Since 64k is an integer, ceil(f * 2^22)
// > 64k iff f * 2^22 > 64k iff f > k * 2^-16, so adding 2^22 - 1 - 64k carries into bit 22 exactly
// when the value rounds up (a ceiling that reaches 2^22 lands on hi, which is also the SR result, as f
// > 1 - 2^-22 exceeds every k * 2^-16).  From a = 6 up the sum is at least 7 << 22, so clamping it to
// (8 << 22) - 1 gives code 7 for every a >= 6 (and for infinities and NaN).
// ---------------------------------------------------------------------------------------------

// Integer multiply-adds written out, so that they stay on the multiply-add pipe.
__device__ __forceinline__ uint32_t mulhi_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.hi.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t mad_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// The rounding above for the two values t0, t1 whose random k are the low and high halves of one Philox
// output word: u = bits(z) + 2^22 - 1 - 64k (64k is a sub-mask of 2^22 - 1), clamped, gives the
// magnitude code u >> 22; bit 3 is the sign of t.  The codes are added to acc0 at nibble n0 and to
// acc1 at nibble n1 (acc0 and acc1 may be the same word).  The integer work is split between the two
// integer pipes: the halves of the word, 64k and the nibble placement as multiply-adds, the sum, the
// clamp, the shift and the sign on the logic pipe (the split measured fastest; Philox's multiplies
// already load the multiply-add pipe).
__device__ __forceinline__ void e2m1_sr_pair(float t0, float t1, uint32_t word, uint32_t& acc0, int n0, uint32_t& acc1,
                                             int n1) {
    const uint32_t r1 = mulhi_u32(word, 0x10000u);                 // high half
    const uint32_t r0 = mad_u32(r1, 0xFFFF0000u, word);             // low half: word - 2^16 r1
    const uint32_t k[2] = {mad_u32(r0, 64u, 0u), mad_u32(r1, 64u, 0u)};
    const float t[2] = {t0, t1};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const uint32_t z = __float_as_uint(__fmul_ru(fabsf(t[e]), __uint_as_float(0x00800000u)));
        const uint32_t u = min((z + 0x3FFFFFu) - k[e], 0x01FFFFFFu);
        const int n = e ? n1 : n0;
        // sign on the logic pipe: code = (u >> 22) | (bit 31 of t >> 28), placed by one multiply-add
        const uint32_t code = (u >> 22) | ((__float_as_uint(t[e]) >> 28) & 8u);
        if (e) acc1 = mad_u32(code, 1u << (4 * n), acc1);
        else acc0 = mad_u32(code, 1u << (4 * n), acc0);
    }
}

// ---------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11): counter (c0..c3), key (k0, k1).
// ---------------------------------------------------------------------------------------------
struct U4 { uint32_t x, y, z, w; };

__device__ __forceinline__ U4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                            uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int rnd = 0; rnd < 10; ++rnd) {
        // the low and high words of each 64-bit product as two 32-bit multiplies (faster here than one
        // widening multiply)
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += 0x9E3779B9u; k1 += 0xBB67AE85u;
    }
    return U4{c0, c1, c2, c3};
}

// Packed two-lane FP32 arithmetic (IEEE round-to-nearest per lane, as the scalar forms): one instruction
// for two lanes' operations, the same lane throughput on the FP32 pipe as the scalar forms.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// In-register 16-point Walsh-Hadamard butterflies with strides 1, 2, 4, 8 (no signs, no 1/4) on packed
// pairs: two independent columns transformed together.
__device__ __forceinline__ void fwht16_unscaled_x2(uint64_t v[16]) {
#pragma unroll
    for (int h = 1; h < 16; h *= 2) {
#pragma unroll
        for (int i = 0; i < 16; i += 2 * h) {
#pragma unroll
            for (int j = i; j < i + h; ++j) {
                const uint64_t a = v[j], b = v[j + h];
                v[j] = f2_add(a, b);
                v[j + h] = f2_sub(a, b);
            }
        }
    }
}



// ---------------------------------------------------------------------------------------------
// NVFP4 block-scale arithmetic (FP32, round to nearest, in the documented order).
// ---------------------------------------------------------------------------------------------

// RN(a / m) for a BF16 value a and a constant m, rm = RN(1 / m): the product a * rm followed by one
// correction step with the exact residual a - q0 * m (Markstein) gives the correctly rounded quotient
// for every finite BF16 a when m is 6, 4 or 2688 (checked exhaustively against the IEEE quotient).
// Infinities and NaN take the IEEE division.
__device__ __forceinline__ float div_bf16_by_const(float a, float m, float rm) {
    if (!(a <= FLT_MAX)) return __fdiv_rn(a, m);
    const float q0 = __fmul_rn(a, rm);
    return __fmaf_rn(__fmaf_rn(-q0, m, a), rm, q0);
}

// S = fp32(amax / 2688) for a BF16 amax.
__device__ __forceinline__ float nvfp4_second_scale(float amax) { return div_bf16_by_const(amax, 2688.0f, 1.0f / 2688.0f); }

// bs = E4M3(fp32(fp32(amax_b / m) / S)) with m = 6 (the block maximum maps to the E2M1 maximum) or,
// for the Four-over-Six alternative, m = 4.
__device__ __forceinline__ uint32_t nvfp4_block_scale_m(float amax_b, float S, float m) {
    if (S == 0.0f) return 0u;
    return cvt_e4m3(__fdiv_rn(__fdiv_rn(amax_b, m), S));
}

// RN(1 / S) for nvfp4_block_scale_fast, or 0 where the fast path does not apply (S zero, below 2^-125,
// or not finite).
__device__ __forceinline__ float nvfp4_fast_rs(float S) {
    return (S >= 1.17549435e-38f * 2.0f && S <= FLT_MAX) ? __frcp_rn(S) : 0.0f;
}

// The same block scale for a BF16 amax_b with rS = nvfp4_fast_rs(S).  fp32(amax_b / m) by the constant
// division above; the quotient by S from y * rS and one Markstein correction, which lands within one unit
// in the last place of fp32(y / S), i.e. within two bit patterns of it (two below a power of two).  E4M3
// rounding is monotone, so when the patterns two below and two above give the same code that is the code
// of fp32(y / S); otherwise (near an E4M3 rounding boundary; 0.07 % of the blocks in a sweep over all BF16
// block and tensor maxima) the IEEE divisions decide.
__device__ __forceinline__ uint32_t nvfp4_block_scale_fast(float amax_b, float S, float rS, float m = 6.0f,
                                                          float rm = 1.0f / 6.0f) {
    if (rS != 0.0f && amax_b <= FLT_MAX) {
        const float y = div_bf16_by_const(amax_b, m, rm);
        const float q0 = __fmul_rn(y, rS);
        const float q = __fmaf_rn(__fmaf_rn(-q0, S, y), rS, q0);
        const uint32_t qb = __float_as_uint(q);
        uint16_t c2;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c2)
            : "f"(__uint_as_float(qb + 2u)), "f"(__uint_as_float(qb >= 2u ? qb - 2u : 0u)));
        const uint32_t lo = c2 & 0xFFu, hi = (uint32_t)c2 >> 8;
        if (lo == hi && lo != 0x7Fu) return lo;
    }
    return nvfp4_block_scale_m(amax_b, S, m);
}

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

// Running max of |bf16| over the two halves of each word in one instruction (max.xorsign.abs: BF16 has
// no flush-to-zero, so subnormals compare exactly; NaN inputs are skipped as in fmax).  The sign bits
// of the result are meaningless: read it through fold_halves or abs_halves.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(acc), "r"(w));
    return d;
}
// The same on the integer pipe (mask, then unsigned 16-bit max; exact magnitudes in the halves), for
// kernels whose floating-point pipe is the busier one.
__device__ __forceinline__ uint32_t absmax_bf16x2_int(uint32_t acc, uint32_t w) {
    return __vmaxu2(acc, w & 0x7FFF7FFFu);
}
__device__ __forceinline__ uint32_t abs_halves(uint32_t m2) { return m2 & 0x7FFF7FFFu; }
// The larger magnitude of the two halves, as BF16 bits in the low 16 bits.
__device__ __forceinline__ uint32_t fold_halves(uint32_t m2) {
    m2 = abs_halves(m2);
    return max(m2 & 0xFFFFu, m2 >> 16);
}

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

// Zero what a grouped quantizer does not write in its scale layout of `tile_bound` 128-row tiles (nct
// 4-column words per row, scale columns a multiple of 4): the padded rows after group g's m_g rows up
// to the end of its last tile, and every tile after the last group's (a contiguous byte range).  The
// work is shared by `nwarps` warps of the grid; this is warp `wid` of them.  The tables come from
// load_group_tables (s_ptile[G] = the total number of group tiles).
__device__ __forceinline__ void zero_grouped_padding(uint8_t* __restrict__ s, const int64_t* s_off, const int* s_ptile,
                                                     int G, int64_t nct, int64_t tile_bound, int64_t wid,
                                                     int64_t nwarps) {
    // (offsets that are not non-decreasing are invalid input; the clamps keep every store inside the
    // layout all the same)
    const int lane = threadIdx.x & 31;
    for (int64_t g = wid; g < G; g += nwarps) {
        const int64_t first = max64(0, (int64_t)s_ptile[g] * 128 + (s_off[g + 1] - s_off[g]));
        const int64_t end = min64((int64_t)s_ptile[g + 1] * 128, tile_bound * 128);   // < 128 rows, one tile
        // lanes over (row, 4-column word) pairs without divisions: 32 / nct rows at a time when nct <= 32
        if (nct <= 32) {
            const int rows_per = 32 / (int)nct;
            const int rr = lane / (int)nct, kc = lane % (int)nct;
            if (rr < rows_per)
                for (int64_t r = first + rr; r < end; r += rows_per)
                    *reinterpret_cast<uint32_t*>(s + sf_offset(r, 4 * kc, nct)) = 0u;
        } else {
            for (int64_t r = first; r < end; ++r)
                for (int64_t c = lane; c < nct; c += 32) *reinterpret_cast<uint32_t*>(s + sf_offset(r, 4 * c, nct)) = 0u;
        }
    }
    const int64_t used = min64(max64(0, (int64_t)s_ptile[G]), tile_bound);
    uint4* tail = reinterpret_cast<uint4*>(s + used * nct * 512);
    const int64_t n16 = (tile_bound - used) * nct * 32;                         // 512-byte tiles as 16-byte words
    for (int64_t i = wid * 32 + lane; i < n16; i += nwarps * 32) tail[i] = make_uint4(0u, 0u, 0u, 0u);
}

// The same for a row r shared by the N lanes [base, base + N) of the warp (lane `sub` of them; N = 16
// or 32, all lanes of the warp calling together): each round the N lanes test N evenly spaced offsets
// of the remaining range and a ballot keeps the span after the last offset <= r, so G = 128 groups take
// two rounds instead of seven dependent steps.
template <int N>
__device__ __forceinline__ int64_t grouped_scale_row_lanes(const int64_t* s_off, const int* s_ptile, int G, int64_t r,
                                                           int sub, int base) {
    int lo = 0, span = G;                              // invariant: s_off[lo] <= r, group in [lo, lo + span)
    // a round count that depends on G only keeps the warp converged for the ballot when the two rows of
    // a warp narrow at different speeds (a finished search repeats as a no-op)
    for (int reach = 1; reach < G; reach *= N) {
        const int step = (span + N - 1) / N;
        const int g = lo + sub * step;
        const bool le = g < lo + span && s_off[g] <= r;
        const uint32_t bits = (__ballot_sync(0xFFFFFFFFu, le) >> base) & (N == 32 ? 0xFFFFFFFFu : ((1u << N) - 1u));
        const int k = 31 - __clz(bits);               // lane 0 always passes (g = lo)
        lo += k * step;
        span = min(step, span - k * step);
    }
    return (int64_t)s_ptile[lo] * 128 + (r - s_off[lo]);
}

}  // namespace mxk

