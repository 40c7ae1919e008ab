/*
 * mxoracle.c -- plain, slow CPU oracle for block-scaled microscaling numerics.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent reference that the
 * CUDA library is checked against.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or constant generator with the CUDA library.
 *
 * Sources (web pages; section names as printed on them):
 *   [Miles]    remio.ai, "Miles Blackwell RL Troca a Uniformidade BF16 por
 *              MXFP8 e NVFP4 Nativos" -- MXFP8 = 32 E4M3 values sharing one
 *              E8M0 scale; NVFP4 = E2M1 values with one E4M3 scale per 16,
 *              under a second FP32 scale computed per token; gate/up quantized
 *              jointly; the bit-exact quantizer contract (section "Um
 *              Quantizador Compartilhado E o Verdadeiro Mecanismo").
 *   [4bitter]  socker-news, "NVFP4 RL training" -- per-token activation scale
 *              ("Baseline recipe details"), dequantized backward
 *              y = x * DQ(Q(w_bf16)).
 *   [E2E]      thelatestinai.com 2610.34915, "End-to-End MXFP8 RL on
 *              Blackwell" -- E8M0 keeps only the exponent (Table 10, F6);
 *              synchronized weights equal the learner's bytes (abstract).
 *   [MaxText]  developer.nvidia.cn, "Train models faster with JAX and MaxText
 *              using NVFP4" -- section "NVFP4 pretraining recipe": 16-element
 *              blocks, E4M3 block scales under a per-tensor FP32 scale, 16x16
 *              2D weight blocks, random Hadamard transform on WGRAD inputs
 *              only, stochastic rounding of gradients.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - Format fields follow the public OCP MX / NVFP4 definitions: E4M3 bias 7,
 *     no infinities, S.1111.111 = NaN (max 448); E2M1 {0,.5,1,1.5,2,3,4,6};
 *     E8M0 = 2^(c-127), c = 255 NaN.
 *   - Rounding to a format is done by enumerating every finite code and
 *     taking the nearest; ties go to the even mantissa LSB; magnitudes above
 *     the maximum clamp to the maximum (satfinite).  The sign is preserved, so
 *     a negative value that rounds to zero encodes as negative zero.
 *   - MXFP8 scale exponent e = floor(log2(block amax)) - 8 (= emax of E4M3),
 *     clamped to [-127, 127]; amax = 0 gives e = -127.
 *   - NVFP4 second-level scale S = amax / (6 * 448) in FP32; block scale
 *     bs = E4M3(amax_b / 6 / S); codes E2M1(x * r), r = 1 / (bs * S), all in
 *     FP32 round-to-nearest in exactly that order; r = 0 when bs * S = 0.
 *   - SR: Philox4x32-10 keyed by the seed, one 16-bit uniform per element.
 *   - RHT: 16-point Sylvester Hadamard, one seeded sign vector, 1/4 scaling.
 *
 * Floating point: compile with -ffp-contract=off and without fast-math; every
 * float operation below is one IEEE binary32 operation rounded to nearest.
 * Where double is used, the value is exact (proved in the comment beside it).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Formats: values decoded from the bit-field definitions.                  */
/* ------------------------------------------------------------------------ */

/* E4M3 (FN): s eeee mmm, bias 7.  e = 0 is subnormal m * 2^-9.  0x7F/0xFF NaN. */
ORC_API double orc_e4m3_value(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* E2M1: s ee m, bias 1.  e = 0 is subnormal m * 0.5. */
ORC_API double orc_e2m1_value(uint8_t c) {
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + m / 2.0, e - 1);
    return s ? -mag : mag;
}

/* E8M0: unsigned exponent, 2^(c - 127); 0xFF NaN. */
ORC_API double orc_e8m0_value(uint8_t c) {
    if (c == 255) return NAN;
    return ldexp(1.0, (int)c - 127);
}

/* Nearest finite code by enumeration over the non-negative codes 0..n-1,
 * ties to the code whose mantissa LSB (bit 0) is 0, magnitude clamped to
 * the largest finite value first (satfinite).  |v| - value is exact in double
 * for every v passed in here (v has at most 24 significant bits and lies
 * within 2^-160..2^9 of the candidates, or is far below the smallest nonzero
 * candidate, in which case zero wins regardless of rounding). */
static uint8_t enumerate_nearest(double a, double (*value)(uint8_t), int ncodes, double maxval) {
    if (a > maxval) a = maxval;
    int best = 0;
    double bestd = fabs(a - value(0));
    for (int c = 1; c < ncodes; ++c) {
        double d = fabs(a - value((uint8_t)c));
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)best;
}

ORC_API uint8_t orc_e4m3_encode(double v) {
    /* codes 0x00..0x7E are the finite non-negative values (0x7F is NaN) */
    uint8_t c = enumerate_nearest(fabs(v), orc_e4m3_value, 127, 448.0);
    return (signbit(v) ? 0x80 : 0x00) | c;
}

ORC_API uint8_t orc_e2m1_encode(double v) {
    uint8_t c = enumerate_nearest(fabs(v), orc_e2m1_value, 8, 6.0);
    return (signbit(v) ? 0x8 : 0x0) | c;
}

/* BF16 bits -> value (exact). */
static float bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* FP32 -> BF16, round to nearest even, by comparing the two neighbouring
 * BF16 values (truncation and the next one away from zero).  The distances
 * are exact in double.  Subnormals need no special case: BF16 shares FP32's
 * exponent range, so both neighbours are plain bit patterns. */
ORC_API uint16_t orc_float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isnan(f)) return 0x7FC0;
    uint32_t lo = u & 0xFFFF0000u, hi = lo + 0x10000u;
    float flo, fhi;
    memcpy(&flo, &lo, 4);
    memcpy(&fhi, &hi, 4);
    double dlo = fabs((double)f - (double)flo), dhi = fabs((double)fhi - (double)f);
    uint32_t pick;
    if (dlo < dhi) pick = lo;
    else if (dhi < dlo) pick = hi;
    else pick = ((lo >> 16) & 1) ? hi : lo;
    return (uint16_t)(pick >> 16);
}

/* ------------------------------------------------------------------------ */
/* Counter-based RNG: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel   */
/* random numbers: as easy as 1, 2, 3", SC'11), written from its definition: */
/* ten rounds of two 32x32->64 multiplies with round keys bumped by the      */
/* Weyl constants between rounds.                                            */
/* ------------------------------------------------------------------------ */
ORC_API void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* 16 random bits for logical element index i under key `seed`:
 * counter = (i>>3 low, i>>3 high, 0, 0); word (i>>1)&3; low half if i even. */
ORC_API uint32_t orc_sr_bits16(uint64_t seed, uint64_t i) {
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint64_t blk = i >> 3;
    uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    uint32_t w = out[(i >> 1) & 3];
    return (i & 1) ? (w >> 16) : (w & 0xFFFFu);
}

/* RHT sign vector: bit j of word 0 of Philox(key = seed, ctr = (0,0,1,0));
 * a set bit means d_j = -1. */
ORC_API void orc_rht16_signs(uint64_t seed, int signs[16]) {
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {0u, 0u, 1u, 0u};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    for (int j = 0; j < 16; ++j) signs[j] = ((out[0] >> j) & 1u) ? -1 : 1;
}

/* ------------------------------------------------------------------------ */
/* GEMM scale-factor layout.  A compact scale matrix [rows, scols] (one byte */
/* per block, blocks along the GEMM's K) is stored as 512-byte tiles of 128  */
/* rows x 4 scale-columns, tiles in row-major order; inside a tile the byte  */
/* for (r, c) is at (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4).  Padding   */
/* (rows up to a multiple of 128, scols up to a multiple of 4) is zero.      */
/* ------------------------------------------------------------------------ */
ORC_API int64_t orc_scale_layout_bytes(int64_t rows, int64_t scols) {
    int64_t rt = (rows + 127) / 128, ct = (scols + 3) / 4;
    return rt * ct * 512;
}

ORC_API int64_t orc_scale_layout_offset(int64_t r, int64_t c, int64_t scols) {
    int64_t ct = (scols + 3) / 4;
    int64_t tile = (r / 128) * ct + (c / 4);
    return tile * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);
}

ORC_API void orc_scales_to_gemm_layout(const uint8_t* compact, int64_t rows, int64_t scols, uint8_t* out) {
    memset(out, 0, (size_t)orc_scale_layout_bytes(rows, scols));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < scols; ++c)
            out[orc_scale_layout_offset(r, c, scols)] = compact[r * scols + c];
}

ORC_API void orc_scales_from_gemm_layout(const uint8_t* laid, int64_t rows, int64_t scols, uint8_t* compact) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < scols; ++c)
            compact[r * scols + c] = laid[orc_scale_layout_offset(r, c, scols)];
}

/* Grouped variant for expert-sorted rows: group g's rows [off[g], off[g+1])
 * are placed from padded row P_g = sum over j < g of ceil(m_j / 128) * 128, so
 * every group starts on a 128-row tile; row r of group g sits at padded row
 * P_g + (r - off[g]) of the plain layout above.  Padding is zero. */
ORC_API int64_t orc_grouped_padded_rows(int64_t G, const int64_t* off) {
    int64_t p = 0;
    for (int64_t g = 0; g < G; ++g) p += (off[g + 1] - off[g] + 127) / 128 * 128;
    return p;
}

ORC_API void orc_scales_to_grouped_layout(const uint8_t* compact, int64_t rows, int64_t scols, int64_t G,
                                          const int64_t* off, uint8_t* out, int64_t out_bytes) {
    memset(out, 0, (size_t)out_bytes);
    int64_t P = 0;
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t r = off[g]; r < off[g + 1]; ++r)
            for (int64_t c = 0; c < scols; ++c)
                out[orc_scale_layout_offset(P + (r - off[g]), c, scols)] = compact[r * scols + c];
        P += (off[g + 1] - off[g] + 127) / 128 * 128;
    }
    (void)rows;
}

/* ------------------------------------------------------------------------ */
/* MXFP8: one E8M0 scale per 32 consecutive elements along the GEMM's K.     */
/* [Miles] "cada bloco de 32 valores E4M3 compartilha uma escala E8M0";      */
/* [E2E] Table 10 F6: E8M0 keeps only the exponent.                          */
/* ------------------------------------------------------------------------ */

/* Quantize one block of n values v[0..n-1] (n = 32).  Returns the E8M0 code,
 * writes E4M3 codes.  Scaling by 2^-e is exact in double (no underflow for
 * BF16 inputs: |v| >= 2^-133 and -e >= -127 keep it above 2^-260). */
static uint8_t mxfp8_block(const double* v, int n, uint8_t* q) {
    double amax = 0.0;
    for (int i = 0; i < n; ++i) amax = fmax(amax, fabs(v[i]));
    int e;
    if (amax == 0.0) {
        e = -127;
    } else {
        int ex;
        frexp(amax, &ex);            /* amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1 */
        e = (ex - 1) - 8;            /* 8 = exponent of E4M3's largest power of two (256) */
        if (e < -127) e = -127;
        if (e > 127) e = 127;
    }
    for (int i = 0; i < n; ++i) q[i] = orc_e4m3_encode(ldexp(v[i], -e));
    return (uint8_t)(e + 127);
}

/* Row-wise: blocks of 32 along cols.  x [rows, ldx] BF16; q [rows, cols];
 * s compact [rows, cols/32]. */
ORC_API void orc_mxfp8_quantize_rowwise(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                                        uint8_t* q, uint8_t* s) {
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double v[32];
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 32; ++i) v[i] = bf16_to_float(x[r * ldx + b * 32 + i]);
            s[r * nb + b] = mxfp8_block(v, 32, q + r * cols + b * 32);
        }
    }
}

/* Column-wise: blocks of 32 along rows, output stored transposed so that the
 * blocks are contiguous along the consuming GEMM's K:  q [cols, rows];
 * s compact [cols, rows/32]. */
ORC_API void orc_mxfp8_quantize_colwise(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                                        uint8_t* q, uint8_t* s) {
    int64_t nb = rows / 32;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < cols; ++c) {
        double v[32];
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 32; ++i) v[i] = bf16_to_float(x[(b * 32 + i) * ldx + c]);
            s[c * nb + b] = mxfp8_block(v, 32, q + c * rows + b * 32);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Blockwise FP8 ([PT page] "FP8 nas camadas lineares": E4M3, weights in     */
/* [128, 128] blocks, input activations and output gradients in [1, 128]     */
/* tiles, one FP32 scale per block; option: power-of-two scales).  Per block */
/* with amax = max |x|:                                                      */
/*   FP32 scale:    s = fp32(amax / 448), q_i = E4M3(fp32(x_i / s));         */
/*                  amax = 0 gives s = 0 and q = 0                           */
/*   power of two:  k = the smallest integer with 448 * 2^k >= amax,         */
/*                  clamped to [-127, 127] (amax = 0 gives -127); s = 2^k;    */
/*                  q_i = E4M3(x_i * 2^-k) (exact scaling, one rounding)     */
/* The power-of-two k is an E8M0 exponent: code k + 127.                     */
/* ------------------------------------------------------------------------ */

static int fp8bw_pow2_exponent(float amax) {
    if (amax == 0.0f) return -127;
    int ex;
    frexp((double)amax, &ex);                      /* amax in [2^(ex-1), 2^ex) */
    /* 448 * 2^(ex-10) = 0.875 * 2^(ex-1) < amax, so the answer is ex - 9 or above */
    int k = ex - 9;
    while (ldexp(448.0, k) < (double)amax) ++k;     /* exact comparisons in double */
    if (k < -127) k = -127;
    if (k > 127) k = 127;
    return k;
}

/* Codes of the n values of one block; returns its FP32 scale, and the E8M0 code in *e8 (power of two). */
static float fp8bw_block(const float* v, int n, int pow2, uint8_t* q, uint8_t* e8) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(v[i]));
    if (pow2) {
        int k = fp8bw_pow2_exponent(amax);
        for (int i = 0; i < n; ++i) q[i] = orc_e4m3_encode(ldexp((double)v[i], -k));
        *e8 = (uint8_t)(k + 127);
        return (float)ldexp(1.0, k);
    }
    *e8 = 0;
    float sc = amax / 448.0f;
    if (amax == 0.0f) {
        for (int i = 0; i < n; ++i) q[i] = orc_e4m3_encode(0.0 * v[i]);
        return 0.0f;
    }
    for (int i = 0; i < n; ++i) {
        float t = v[i] / sc;
        q[i] = orc_e4m3_encode((double)t);
    }
    return sc;
}

/* Activations / gradients, [1, 128] tiles along K.  x [R, ldx] BF16, K % 128 == 0; q [R, K];
 * s [R, K/128] FP32; e8 [R, K/128] (E8M0 codes of the power-of-two scales, 0 otherwise). */
ORC_API void orc_fp8_blockwise_1x128(const uint16_t* x, int64_t R, int64_t K, int64_t ldx, int pow2,
                                     uint8_t* q, float* s, uint8_t* e8) {
    int64_t nb = K / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        float v[128];
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 128; ++i) v[i] = bf16_to_float(x[r * ldx + b * 128 + i]);
            s[r * nb + b] = fp8bw_block(v, 128, pow2, q + r * K + b * 128, e8 + r * nb + b);
        }
    }
}

/* Weights, [128, 128] blocks (the last block row / column may be partial).  w [O, H] BF16;
 * q_row [O, H]; q_col [H, O] (the same codes, transposed); s [ceil(O/128), ceil(H/128)] FP32; e8 the
 * same shape (E8M0 codes of the power-of-two scales, 0 otherwise). */
ORC_API void orc_fp8_blockwise_128x128(const uint16_t* w, int64_t O, int64_t H, int pow2,
                                       uint8_t* q_row, uint8_t* q_col, float* s, uint8_t* e8) {
    int64_t bo_n = (O + 127) / 128, bh_n = (H + 127) / 128;
#pragma omp parallel for schedule(static)
    for (int64_t bo = 0; bo < bo_n; ++bo) {
        float* v = (float*)malloc(sizeof(float) * 128 * 128);
        uint8_t* c = (uint8_t*)malloc(128 * 128);
        for (int64_t bh = 0; bh < bh_n; ++bh) {
            int64_t ro = bo * 128, rh = bh * 128;
            int no = (int)(O - ro < 128 ? O - ro : 128), nh = (int)(H - rh < 128 ? H - rh : 128);
            for (int i = 0; i < no; ++i)
                for (int j = 0; j < nh; ++j) v[i * nh + j] = bf16_to_float(w[(ro + i) * H + rh + j]);
            s[bo * bh_n + bh] = fp8bw_block(v, no * nh, pow2, c, e8 + bo * bh_n + bh);
            for (int i = 0; i < no; ++i)
                for (int j = 0; j < nh; ++j) {
                    q_row[(ro + i) * H + rh + j] = c[i * nh + j];
                    q_col[(rh + j) * O + ro + i] = c[i * nh + j];
                }
        }
        free(v);
        free(c);
    }
}

/* ------------------------------------------------------------------------ */
/* NVFP4: E2M1 values, one E4M3 scale per 16, under an FP32 second-level     */
/* scale S ([Miles] per token; [MaxText] per tensor).  For every block:      */
/*   bs = E4M3( fp32( fp32(amax_b / 6) / S ) )      (S = 0 gives bs = 0)     */
/*   d  = fp32( value(bs) * S )                                              */
/*   r  = d == 0 ? 0 : min( fp32(1 / d), FLT_MAX )                           */
/*   q_i = E2M1( fp32(x_i * r) )            -- or SR of fp32(x_i * r)        */
/* ------------------------------------------------------------------------ */

static const float NVFP4_S_DIV = 2688.0f;   /* 6 * 448: E2M1 max times E4M3 max */

ORC_API float orc_nvfp4_second_scale(float amax) { return amax / NVFP4_S_DIV; }

ORC_API uint8_t orc_nvfp4_block_scale(float amax_b, float S) {
    if (S == 0.0f) return 0;
    float t = amax_b / 6.0f;
    t = t / S;
    return orc_e4m3_encode((double)t);
}

ORC_API float orc_nvfp4_block_recip(uint8_t bs, float S) {
    float d = (float)orc_e4m3_value(bs) * S;
    if (d == 0.0f) return 0.0f;
    float r = 1.0f / d;
    return r > FLT_MAX ? FLT_MAX : r;
}

/* Stochastic rounding of a finite float v onto the E2M1 grid with 16 random
 * bits k: a = |v|; a >= 6 -> 6; otherwise lo = the largest grid value <= a,
 * hi = the next, f = (a - lo) / (hi - lo) (exact: Sterbenz, and hi - lo is a
 * power of two); round up iff f > k * 2^-16.  The sign is reapplied. */
ORC_API uint8_t orc_e2m1_encode_sr(float v, uint32_t k16) {
    static const float grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    float a = fabsf(v);
    uint8_t code;
    if (a >= 6.0f) {
        code = 7;
    } else {
        int lo = 0;
        for (int c = 0; c < 8; ++c)
            if (grid[c] <= a) lo = c;
        float f = (a - grid[lo]) / (grid[lo + 1] - grid[lo]);
        float u = (float)k16 * (1.0f / 65536.0f);
        code = (uint8_t)(f > u ? lo + 1 : lo);
    }
    return (signbit(v) ? 0x8 : 0x0) | code;
}

static void put_nibble(uint8_t* row, int64_t k, uint8_t code) {
    /* two codes per byte, the even index in the low nibble */
    if (k & 1) row[k >> 1] = (uint8_t)((row[k >> 1] & 0x0F) | (code << 4));
    else       row[k >> 1] = (uint8_t)((row[k >> 1] & 0xF0) | (code & 0x0F));
}

/* Per-token 1x16 quantization ([Miles] "calcula uma escala de ativacao FP32
 * por token online"; [4bitter] per-token activation scaling).
 * x [T, ldx] BF16; q [T, H/2]; s compact [T, H/16]; s_tok [T]. */
ORC_API void orc_nvfp4_quantize_per_token(const uint16_t* x, int64_t T, int64_t H, int64_t ldx,
                                          uint8_t* q, uint8_t* s, float* s_tok) {
    int64_t nb = H / 16;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t* xr = x + t * ldx;
        float amax = 0.0f;
        for (int64_t k = 0; k < H; ++k) amax = fmaxf(amax, fabsf(bf16_to_float(xr[k])));
        float S = orc_nvfp4_second_scale(amax);
        s_tok[t] = S;
        uint8_t* qr = q + t * (H / 2);
        for (int64_t b = 0; b < nb; ++b) {
            float ab = 0.0f;
            for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(bf16_to_float(xr[b * 16 + i])));
            uint8_t bs = orc_nvfp4_block_scale(ab, S);
            float r = orc_nvfp4_block_recip(bs, S);
            s[t * nb + b] = bs;
            for (int i = 0; i < 16; ++i) {
                float v = bf16_to_float(xr[b * 16 + i]) * r;
                put_nibble(qr, b * 16 + i, orc_e2m1_encode((double)v));
            }
        }
    }
}

/* 16x16 2D weight quantization ([MaxText] "2D weight scaling": one FP8
 * scale per 16x16 block so FPROP and the transposed DGRAD see the same
 * values; per-tensor FP32 second level).  One matrix w [O, H] (gate and up
 * stacked when they share a scale, [Miles]).
 * q_row [O, H/2] (blocks along H); q_col [H, O/2] (the same codes,
 * transposed); s_tile compact [O/16, H/16]; *s_w the FP32 scale. */
ORC_API void orc_nvfp4_quantize_weight_2d(const uint16_t* w, int64_t O, int64_t H,
                                          uint8_t* q_row, uint8_t* q_col, uint8_t* s_tile, float* s_w) {
    float amax = 0.0f;
    for (int64_t i = 0; i < O * H; ++i) amax = fmaxf(amax, fabsf(bf16_to_float(w[i])));
    float S = orc_nvfp4_second_scale(amax);
    *s_w = S;
    int64_t to = O / 16, th = H / 16;
#pragma omp parallel for schedule(static)
    for (int64_t bo = 0; bo < to; ++bo) {
        for (int64_t bh = 0; bh < th; ++bh) {
            float ab = 0.0f;
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j)
                    ab = fmaxf(ab, fabsf(bf16_to_float(w[(bo * 16 + i) * H + bh * 16 + j])));
            uint8_t bs = orc_nvfp4_block_scale(ab, S);
            float r = orc_nvfp4_block_recip(bs, S);
            s_tile[bo * th + bh] = bs;
            for (int i = 0; i < 16; ++i) {
                for (int j = 0; j < 16; ++j) {
                    int64_t o = bo * 16 + i, h = bh * 16 + j;
                    float v = bf16_to_float(w[o * H + h]) * r;
                    uint8_t c = orc_e2m1_encode((double)v);
                    put_nibble(q_row + o * (H / 2), h, c);
                    put_nibble(q_col + h * (O / 2), o, c);
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Four-over-Six ([NVIDIA RL blog] "Four-Over-Six (4/6)": instead of always  */
/* mapping a block's maximum to the E2M1 maximum 6, map it to 4 or to 6 and  */
/* keep the lower error; the largest error drops from 1/6 to 1/8 of the      */
/* range).  Readings: the error is the largest absolute difference between   */
/* a value and its FP32 dequantization fp32(fp32(value(q) * value(bs)) * S); */
/* 4 is kept only if strictly better (ties keep the standard 6); S is        */
/* unchanged (amax / 2688), so consumers of the codes need no change.        */
/*   bs_m = E4M3( fp32( fp32(amax_b / m) / S ) ),  m in {6, 4}               */
/* ------------------------------------------------------------------------ */

static uint8_t nvfp4_block_scale_m(float amax_b, float S, float m) {
    if (S == 0.0f) return 0;
    float t = amax_b / m;
    t = t / S;
    return orc_e4m3_encode((double)t);
}

/* Codes of n values under block scale bs and second-level scale S, and the largest absolute
 * dequantization error. */
static float nvfp4_block_candidate(const float* x, int n, uint8_t bs, float S, uint8_t* codes) {
    float r = orc_nvfp4_block_recip(bs, S);
    float bsv = (float)orc_e4m3_value(bs);
    float err = 0.0f;
    for (int i = 0; i < n; ++i) {
        float v = x[i] * r;
        codes[i] = orc_e2m1_encode((double)v);
        float prod = (float)orc_e2m1_value(codes[i]) * bsv;
        float deq = prod * S;
        err = fmaxf(err, fabsf(deq - x[i]));
    }
    return err;
}

/* Chooses between the two candidates for one block of n values (n = 16 or 256); returns the scale,
 * the codes in codes[]. */
static uint8_t nvfp4_block_four_over_six(const float* x, int n, float amax_b, float S, uint8_t* codes) {
    uint8_t c6[256], c4[256];
    uint8_t bs6 = nvfp4_block_scale_m(amax_b, S, 6.0f);
    uint8_t bs4 = nvfp4_block_scale_m(amax_b, S, 4.0f);
    float e6 = nvfp4_block_candidate(x, n, bs6, S, c6);
    float e4 = nvfp4_block_candidate(x, n, bs4, S, c4);
    int four = e4 < e6;
    memcpy(codes, four ? c4 : c6, (size_t)n);
    return four ? bs4 : bs6;
}

/* Per-token 1x16 with 4/6 block scales; arguments as orc_nvfp4_quantize_per_token. */
ORC_API void orc_nvfp4_quantize_per_token_46(const uint16_t* x, int64_t T, int64_t H, int64_t ldx,
                                             uint8_t* q, uint8_t* s, float* s_tok) {
    int64_t nb = H / 16;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t* xr = x + t * ldx;
        float amax = 0.0f;
        for (int64_t k = 0; k < H; ++k) amax = fmaxf(amax, fabsf(bf16_to_float(xr[k])));
        float S = orc_nvfp4_second_scale(amax);
        s_tok[t] = S;
        uint8_t* qr = q + t * (H / 2);
        for (int64_t b = 0; b < nb; ++b) {
            float xv[16], ab = 0.0f;
            for (int i = 0; i < 16; ++i) {
                xv[i] = bf16_to_float(xr[b * 16 + i]);
                ab = fmaxf(ab, fabsf(xv[i]));
            }
            uint8_t codes[16];
            s[t * nb + b] = nvfp4_block_four_over_six(xv, 16, ab, S, codes);
            for (int i = 0; i < 16; ++i) put_nibble(qr, b * 16 + i, codes[i]);
        }
    }
}

/* 16x16 2D weights with 4/6 tile scales; arguments as orc_nvfp4_quantize_weight_2d.  A tile's values
 * are taken row by row (the error is a maximum, so the order does not matter). */
ORC_API void orc_nvfp4_quantize_weight_2d_46(const uint16_t* w, int64_t O, int64_t H,
                                             uint8_t* q_row, uint8_t* q_col, uint8_t* s_tile, float* s_w) {
    float amax = 0.0f;
    for (int64_t i = 0; i < O * H; ++i) amax = fmaxf(amax, fabsf(bf16_to_float(w[i])));
    float S = orc_nvfp4_second_scale(amax);
    *s_w = S;
    int64_t to = O / 16, th = H / 16;
#pragma omp parallel for schedule(static)
    for (int64_t bo = 0; bo < to; ++bo) {
        for (int64_t bh = 0; bh < th; ++bh) {
            float xv[256], ab = 0.0f;
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j) {
                    xv[i * 16 + j] = bf16_to_float(w[(bo * 16 + i) * H + bh * 16 + j]);
                    ab = fmaxf(ab, fabsf(xv[i * 16 + j]));
                }
            uint8_t codes[256];
            s_tile[bo * th + bh] = nvfp4_block_four_over_six(xv, 256, ab, S, codes);
            for (int i = 0; i < 16; ++i) {
                for (int j = 0; j < 16; ++j) {
                    int64_t o = bo * 16 + i, h = bh * 16 + j;
                    put_nibble(q_row + o * (H / 2), h, codes[i * 16 + j]);
                    put_nibble(q_col + h * (O / 2), o, codes[i * 16 + j]);
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Random Hadamard transform ([MaxText]: applied only to WGRAD inputs).      */
/* Along the token dim, per column and per aligned 16-token chunk:           */
/*   v = d * x (exact sign flip); Walsh-Hadamard butterflies with strides    */
/*   1, 2, 4, 8, (a, b) -> (a + b, a - b) in FP32; y = BF16_RNE(v / 4).      */
/* ------------------------------------------------------------------------ */
static void rht16_vec(const float in[16], const int signs[16], float out[16]) {
    float v[16];
    for (int j = 0; j < 16; ++j) v[j] = signs[j] < 0 ? -in[j] : in[j];
    for (int h = 1; h < 16; h *= 2)
        for (int i = 0; i < 16; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
    for (int j = 0; j < 16; ++j) out[j] = v[j] * 0.25f;
}

/* Exposed for the oracle's own tests: the FP32 transform before BF16. */
ORC_API void orc_rht16_vec_f32(const float* in, uint64_t seed, float* out) {
    int signs[16];
    orc_rht16_signs(seed, signs);
    rht16_vec(in, signs, out);
}

/* x, y [T, N] BF16. */
ORC_API void orc_rht16(const uint16_t* x, int64_t T, int64_t N, uint64_t seed, uint16_t* y) {
    int signs[16];
    orc_rht16_signs(seed, signs);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t c = 0; c < T / 16; ++c) {
            float in[16], out[16];
            for (int j = 0; j < 16; ++j) in[j] = bf16_to_float(x[(c * 16 + j) * N + n]);
            rht16_vec(in, signs, out);
            for (int j = 0; j < 16; ++j) y[(c * 16 + j) * N + n] = orc_float_to_bf16(out[j]);
        }
    }
}

/* 1x16 quantization with a per-tensor FP32 second-level scale ([MaxText]), in its two passes.
 * Pass 1 (orc_nvfp4_1x16_amax): A = amax over the (BF16-rounded, transformed) tensor.  The RHT acts
 * on each column separately, so the amax of a tensor is the max over any split into column slabs.
 * Pass 2 (orc_nvfp4_1x16_pass2): with S = A / 2688, per block as in the per-token case, RNE, or SR
 * with the 16 bits of logical element i = t * N_total + n_global.  The slab holds columns
 * [n_offset, n_offset + N) of a [T, N_total] tensor.
 * colwise = 1: blocks of 16 along T, output transposed q [N, T/2], s compact [N, T/16].
 * colwise = 0: blocks along N, q [T, N/2], s compact [T, N/16] (rht must be 0). */
ORC_API float orc_nvfp4_1x16_amax(const uint16_t* x, int64_t T, int64_t N, int rht, uint64_t rht_seed) {
    uint16_t* y = NULL;
    const uint16_t* src = x;
    if (rht) {
        y = (uint16_t*)malloc((size_t)(T * N) * sizeof(uint16_t));
        orc_rht16(x, T, N, rht_seed, y);
        src = y;
    }
    float amax = 0.0f;
    for (int64_t i = 0; i < T * N; ++i) amax = fmaxf(amax, fabsf(bf16_to_float(src[i])));
    free(y);
    return amax;
}

ORC_API void orc_nvfp4_1x16_pass2(const uint16_t* x, int64_t T, int64_t N, int64_t n_offset, int64_t N_total,
                                  int colwise, int rht, uint64_t rht_seed, int sr, uint64_t sr_seed, float S,
                                  uint8_t* q, uint8_t* s) {
    uint16_t* y = NULL;
    const uint16_t* src = x;
    if (rht) {
        y = (uint16_t*)malloc((size_t)(T * N) * sizeof(uint16_t));
        orc_rht16(x, T, N, rht_seed, y);
        src = y;
    }
    if (colwise) {
        int64_t nb = T / 16;
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t b = 0; b < nb; ++b) {
                float ab = 0.0f;
                for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(bf16_to_float(src[(b * 16 + i) * N + n])));
                uint8_t bs = orc_nvfp4_block_scale(ab, S);
                float r = orc_nvfp4_block_recip(bs, S);
                s[n * nb + b] = bs;
                for (int i = 0; i < 16; ++i) {
                    int64_t t = b * 16 + i;
                    float v = bf16_to_float(src[t * N + n]) * r;
                    uint64_t gi = (uint64_t)(t * N_total + n_offset + n);
                    uint8_t c = sr ? orc_e2m1_encode_sr(v, orc_sr_bits16(sr_seed, gi)) : orc_e2m1_encode((double)v);
                    put_nibble(q + n * (T / 2), t, c);
                }
            }
        }
    } else {
        int64_t nb = N / 16;
#pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t b = 0; b < nb; ++b) {
                float ab = 0.0f;
                for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(bf16_to_float(src[t * N + b * 16 + i])));
                uint8_t bs = orc_nvfp4_block_scale(ab, S);
                float r = orc_nvfp4_block_recip(bs, S);
                s[t * nb + b] = bs;
                for (int i = 0; i < 16; ++i) {
                    int64_t n = b * 16 + i;
                    float v = bf16_to_float(src[t * N + n]) * r;
                    uint64_t gi = (uint64_t)(t * N_total + n_offset + n);
                    uint8_t c = sr ? orc_e2m1_encode_sr(v, orc_sr_bits16(sr_seed, gi)) : orc_e2m1_encode((double)v);
                    put_nibble(q + t * (N / 2), n, c);
                }
            }
        }
    }
    free(y);
}

/* Both passes on a whole [T, N] tensor. */
ORC_API void orc_nvfp4_quantize_1x16(const uint16_t* x, int64_t T, int64_t N, int colwise, int rht,
                                     uint64_t rht_seed, int sr, uint64_t sr_seed,
                                     uint8_t* q, uint8_t* s, float* s_tensor) {
    float S = orc_nvfp4_second_scale(orc_nvfp4_1x16_amax(x, T, N, rht, rht_seed));
    *s_tensor = S;
    orc_nvfp4_1x16_pass2(x, T, N, 0, N, colwise, rht, rht_seed, sr, sr_seed, S, q, s);
}

/* ------------------------------------------------------------------------ */
/* Dequantize to BF16 ([4bitter] dequantized backward y = x * DQ(Q(w)):      */
/* the backward operand is rebuilt from the exact forward values).           */
/*   MXFP8: y = BF16_RNE(value(q) * 2^e)          (the product is exact)     */
/*   NVFP4: y = BF16_RNE(fp32(value(q) * value(bs)) * S)                     */
/* ------------------------------------------------------------------------ */

/* q [R, K]; s compact [R, K/32]; y [R, K] BF16.  value(q) * 2^e has at most
 * 4 significant bits and lies in [2^-136, 2^128), so it is exact in FP32. */
ORC_API void orc_dequant_mxfp8(const uint8_t* q, const uint8_t* s, int64_t R, int64_t K, uint16_t* y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k) {
            double v = orc_e4m3_value(q[r * K + k]) * orc_e8m0_value(s[r * (K / 32) + k / 32]);
            y[r * K + k] = orc_float_to_bf16((float)v);
        }
}

/* q [R, K/2] packed; s compact [R, K/16]; s2 per row (s2_per_row = 1) or a
 * single per-tensor value; y [R, K] BF16. */
ORC_API void orc_dequant_nvfp4(const uint8_t* q, const uint8_t* s, const float* s2, int s2_per_row,
                               int64_t R, int64_t K, uint16_t* y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        float S = s2_per_row ? s2[r] : s2[0];
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = q[r * (K / 2) + k / 2];
            uint8_t code = (k & 1) ? (byte >> 4) : (byte & 0xF);
            float p = (float)(orc_e2m1_value(code) * orc_e4m3_value(s[r * (K / 16) + k / 16]));
            y[r * K + k] = orc_float_to_bf16(p * S);
        }
    }
}

/* Exact decoded values in double, for the FP64 GEMM reference.
 * MXFP8: value(q) * 2^e.  NVFP4: value(q) * value(bs) (second level not
 * applied; the reference multiplies it in separately). */
ORC_API void orc_decode_mxfp8_f64(const uint8_t* q, const uint8_t* s, int64_t R, int64_t K, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k)
            out[r * K + k] = orc_e4m3_value(q[r * K + k]) * orc_e8m0_value(s[r * (K / 32) + k / 32]);
}

ORC_API void orc_decode_nvfp4_f64(const uint8_t* q, const uint8_t* s, int64_t R, int64_t K, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = q[r * (K / 2) + k / 2];
            uint8_t code = (k & 1) ? (byte >> 4) : (byte & 0xF);
            out[r * K + k] = orc_e2m1_value(code) * orc_e4m3_value(s[r * (K / 16) + k / 16]);
        }
}

ORC_API void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

ORC_API int orc_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
