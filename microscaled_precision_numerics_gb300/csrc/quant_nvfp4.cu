// quant_nvfp4.cu -- NVFP4 quantizers (E2M1 values, one E4M3 scale per 16, FP32 second level).
//
//   per-token 1x16 (Miles page: per-token FP32 scale computed online and fused into the activation
//                   quantizer; NVFP4 RL page, "Baseline recipe details")
//   per-tensor 1x16, row-wise or column-wise along tokens, optional RHT, RNE or SR (MaxText page,
//                   "NVFP4 pretraining recipe": 1x16 activations/gradients, RHT on WGRAD inputs,
//                   SR on gradients)
//   standalone RHT16 along tokens
//   16x16 2D weights, both orientations (MaxText page: 2D weight scaling; Miles page: joint gate/up)
//
// All scale arithmetic is FP32 round-to-nearest in the documented order (mx_device.cuh); E2M1 and
// E4M3 codes come from the cvt.rn.satfinite instructions, or from the ALU stochastic rounding.
#include "mx_internal.h"

namespace mxk {

namespace {

// ------------------------------------------------------------------------------------------------
// Row-wise 1x16 with a per-token scale.  One warp per row (grid-stride over rows); lane l owns
// the 16-element blocks l, l + 32, ..., so the block-scale arithmetic runs once per 16 elements.
// Rows of up to 32 * RW_MAXB blocks stay in registers between the amax and the quantize pass;
// longer rows are read twice (the second read hits L1/L2).
// ------------------------------------------------------------------------------------------------
constexpr int RW_WARPS = 8;
constexpr int RW_MAXB = 4;     // blocks per lane kept in registers (H <= 2048)
constexpr int RW_CTAS_PER_SM = 4;   // 64 registers: resident warps hide the block-scale division chains

// Quantize one 16-element block held in two 16-byte words; returns the 8 code bytes.
template <bool SR>
__device__ __forceinline__ uint2 quant_block16(const uint4& a, const uint4& b, float r, uint64_t elem0,
                                               uint32_t k0, uint32_t k1) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = __fmul_rn(bf16_lo(w[i]), r);
        v[2 * i + 1] = __fmul_rn(bf16_hi(w[i]), r);
    }
    if (SR) {
        // elements elem0 .. elem0 + 15 (elem0 % 16 == 0): two Philox blocks of 8
        uint32_t c[2] = {0u, 0u};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint64_t blk = (elem0 >> 3) + h;
            const U4 rnd = philox4x32_10((uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u, k0, k1);
            const uint32_t rw[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
#pragma unroll
            for (int jp = 0; jp < 4; ++jp)
                e2m1_sr_pair(v[8 * h + 2 * jp], v[8 * h + 2 * jp + 1], rw[jp], c[h], 2 * jp, c[h], 2 * jp + 1);
        }
        return make_uint2(c[0], c[1]);
    }
    return make_uint2(cvt_e2m1x8(v), cvt_e2m1x8(v + 8));
}

// Largest |fp32(fp32(value(q_i) * value(bs)) * S) - x_i| over n values (n a multiple of 8) whose codes are
// packed 8 per word (even index in the low nibble).  value(q) * value(bs) has at most 6 significant bits
// and lies in [2^-10, 2688], so the product of the two FP16 decodes (two elements per instruction: the
// hardware E2M1 and E4M3 conversions, and a packed FP16 multiply) is exact and equals the FP32 product.
__device__ __forceinline__ float nvfp4_max_dq_error(const float* x, const uint32_t* codes, int n, uint32_t bs, float S) {
    uint32_t bs2;                                       // value(bs) in both FP16 halves
    asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(bs2) : "r"((bs & 0xFFu) * 0x101u));
    float err = 0.0f;
#pragma unroll
    for (int i = 0; i < n; i += 2) {
        const uint32_t q2 = e2m1x2_to_f16x2(codes[i >> 3] >> (4 * (i & 7)));
        uint32_t p2;
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p2) : "r"(q2), "r"(bs2));
        const float p0 = __half2float(__ushort_as_half((unsigned short)(p2 & 0xFFFFu)));
        const float p1 = __half2float(__ushort_as_half((unsigned short)(p2 >> 16)));
        err = fmaxf(err, fabsf(__fsub_rn(__fmul_rn(p0, S), x[i])));
        err = fmaxf(err, fabsf(__fsub_rn(__fmul_rn(p1, S), x[i + 1])));
    }
    return err;
}

// Four-over-Six (NVIDIA RL blog, "Four-Over-Six (4/6)"): the block is quantized with its maximum mapped
// to 6 and to 4, and the candidate with the smaller largest dequantization error is kept (a tie keeps
// 6).  Returns the 8 code bytes and the chosen scale.
__device__ __forceinline__ uint2 quant_block16_46(const uint4& a, const uint4& c, float amax_b, float S, float rS,
                                                  uint32_t& bs_out) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
    float x[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) { x[2 * i] = bf16_lo(w[i]); x[2 * i + 1] = bf16_hi(w[i]); }
    uint32_t best[2], bs_best = 0;
    float err_best = 0.0f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t bs = k == 0 ? nvfp4_block_scale_fast(amax_b, S, rS) : nvfp4_block_scale_fast(amax_b, S, rS, 4.0f, 0.25f);
        const float r = nvfp4_block_recip(bs, S);
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(x[i], r);
        const uint32_t codes[2] = {cvt_e2m1x8(v), cvt_e2m1x8(v + 8)};
        const float err = nvfp4_max_dq_error(x, codes, 16, bs, S);
        if (k == 0 || err < err_best) { best[0] = codes[0]; best[1] = codes[1]; bs_best = bs; err_best = err; }
    }
    bs_out = bs_best;
    return make_uint2(best[0], best[1]);
}

template <bool GROUPED, int LPR, bool FOUR_SIX = false>
__global__ void __launch_bounds__(RW_WARPS * 32, RW_CTAS_PER_SM)
nvfp4_rowwise_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t H, int64_t ldx,
                     uint8_t* __restrict__ q, uint8_t* __restrict__ s, float* __restrict__ s_tok,
                     int G, const int64_t* __restrict__ group_offsets, bool zero_pad) {
    // LPR lanes per row (32 or 16): a warp works on 32 / LPR rows at once
    constexpr int RPW = 32 / LPR;
    extern __shared__ __align__(16) uint8_t rw_sm[];
    int64_t* s_off = reinterpret_cast<int64_t*>(rw_sm);
    int* s_ptile = reinterpret_cast<int*>(rw_sm + 8 * (G + 1));
    int* s_warp = s_ptile + (G + 1);
    if (GROUPED) load_group_tables(group_offsets, G, s_off, s_ptile, s_warp);

    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR;                      // lane within the row group
    const int half = lane / LPR;                     // which of the warp's rows
    const uint32_t gmask = LPR == 32 ? 0xFFFFFFFFu : (0xFFFFu << (16 * half));
    const int64_t nblk = H / 16;
    const int64_t nct = sf_col_tiles(H, 16);
    const bool cached = nblk <= LPR * RW_MAXB;
    for (int64_t tw = ((int64_t)blockIdx.x * RW_WARPS + (threadIdx.x >> 5)) * RPW; tw < T;
         tw += (int64_t)gridDim.x * RW_WARPS * RPW) {
        const int64_t t = tw + half;
        const bool row_ok = t < T;                   // the warp stays converged for the shuffles below
        const uint4* xr = reinterpret_cast<const uint4*>(x + (row_ok ? t : tw) * ldx);
        uint4 ra[RW_MAXB], rb[RW_MAXB];
        uint32_t bam[RW_MAXB];                       // block amax bits of the cached blocks
        float S;
        if (cached) {
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < RW_MAXB; ++i) {
                const int64_t b = sub + LPR * i;
                ra[i] = rb[i] = make_uint4(0u, 0u, 0u, 0u);
                if (row_ok && b < nblk) { ra[i] = __ldcs(xr + 2 * b); rb[i] = __ldcs(xr + 2 * b + 1); }
                uint32_t m2 = 0;
                m2 = absmax_bf16x2(m2, ra[i].x); m2 = absmax_bf16x2(m2, ra[i].y);
                m2 = absmax_bf16x2(m2, ra[i].z); m2 = absmax_bf16x2(m2, ra[i].w);
                m2 = absmax_bf16x2(m2, rb[i].x); m2 = absmax_bf16x2(m2, rb[i].y);
                m2 = absmax_bf16x2(m2, rb[i].z); m2 = absmax_bf16x2(m2, rb[i].w);
                bam[i] = fold_halves(m2);
                m = max(m, bam[i]);
            }
            const uint32_t amax16 = __reduce_max_sync(gmask, m);
            S = nvfp4_second_scale(__uint_as_float(amax16 << 16));
            if (row_ok && sub == 0) s_tok[t] = S;
        } else {
            uint32_t m2 = 0;
            if (row_ok) {
                for (int64_t b = sub; b < nblk; b += LPR) {
                    const uint4 a = __ldg(xr + 2 * b), c = __ldg(xr + 2 * b + 1);
                    m2 = absmax_bf16x2(m2, a.x); m2 = absmax_bf16x2(m2, a.y);
                    m2 = absmax_bf16x2(m2, a.z); m2 = absmax_bf16x2(m2, a.w);
                    m2 = absmax_bf16x2(m2, c.x); m2 = absmax_bf16x2(m2, c.y);
                    m2 = absmax_bf16x2(m2, c.z); m2 = absmax_bf16x2(m2, c.w);
                }
            }
            const uint32_t amax16 = __reduce_max_sync(gmask, fold_halves(m2));
            S = nvfp4_second_scale(__uint_as_float(amax16 << 16));
            if (row_ok && sub == 0) s_tok[t] = S;
        }
        int64_t srow = t;
        bool srow_ok = true;
        if (GROUPED) {
            srow = grouped_scale_row_lanes<LPR>(s_off, s_ptile, G, row_ok ? t : T - 1, sub, half * LPR);
            srow_ok = srow >= 0 && srow < T + 127 * (int64_t)G;   // stays inside the layout (offsets not checked)
        }
        const float rS = nvfp4_fast_rs(S);

        // codes, and the four consecutive block scales of lanes 4m .. 4m+3 of the row group as one word
        auto emit = [&](int64_t b, bool valid, const uint4& a, const uint4& c, uint32_t bs, float r, uint32_t amax_bits) {
            uint2 codes;
            if (FOUR_SIX) codes = quant_block16_46(a, c, __uint_as_float(amax_bits << 16), S, rS, bs);
            else codes = quant_block16<false>(a, c, r, 0, 0u, 0u);
            if (valid) __stcs(reinterpret_cast<uint2*>(q + t * (H / 2) + b * 8), codes);
            const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, bs, 1);
            const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, bs, 2);
            const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, bs, 3);
            if (valid && srow_ok && (b & 3) == 0) {
                uint8_t* p = s + sf_offset(srow, b, nct);
                if (b + 4 <= nblk) {
                    *reinterpret_cast<uint32_t*>(p) = bs | (b1 << 8) | (b2 << 16) | (b3 << 24);
                } else {
                    const uint32_t bb[4] = {bs, b1, b2, b3};
                    for (int k = 0; k < (int)(nblk - b); ++k) p[k] = (uint8_t)bb[k];
                }
            }
        };
        if (cached) {
            // all block scales first: the lane's independent scale chains overlap
            uint32_t bsv[RW_MAXB];
            float rv[RW_MAXB];
#pragma unroll
            for (int i = 0; i < RW_MAXB; ++i) {
                bsv[i] = FOUR_SIX ? 0u : nvfp4_block_scale_fast(__uint_as_float(bam[i] << 16), S, rS);
                rv[i] = FOUR_SIX ? 0.0f : nvfp4_block_recip(bsv[i], S);
            }
            const int64_t nrounds = (nblk + LPR - 1) / LPR;
#pragma unroll
            for (int i = 0; i < RW_MAXB; ++i) {
                if (i < nrounds) {                  // warp-uniform
                    const int64_t b = sub + LPR * i;
                    emit(b, row_ok && b < nblk, ra[i], rb[i], bsv[i], rv[i], bam[i]);
                }
            }
        } else {
            const int64_t nrounds = (nblk + LPR - 1) / LPR;
            for (int64_t i = 0; i < nrounds; ++i) {
                const int64_t b = sub + LPR * i;
                const bool valid = row_ok && b < nblk;
                uint4 a = make_uint4(0u, 0u, 0u, 0u), c = make_uint4(0u, 0u, 0u, 0u);
                if (valid) { a = __ldcs(xr + 2 * b); c = __ldcs(xr + 2 * b + 1); }
                uint32_t m2 = 0;
                m2 = absmax_bf16x2(m2, a.x); m2 = absmax_bf16x2(m2, a.y); m2 = absmax_bf16x2(m2, a.z); m2 = absmax_bf16x2(m2, a.w);
                m2 = absmax_bf16x2(m2, c.x); m2 = absmax_bf16x2(m2, c.y); m2 = absmax_bf16x2(m2, c.z); m2 = absmax_bf16x2(m2, c.w);
                const uint32_t am = fold_halves(m2);
                const uint32_t bs = FOUR_SIX ? 0u : nvfp4_block_scale_fast(__uint_as_float(am << 16), S, rS);
                emit(b, valid, a, c, bs, FOUR_SIX ? 0.0f : nvfp4_block_recip(bs, S), am);
            }
        }
    }
    if (GROUPED && zero_pad)
        zero_grouped_padding(s, s_off, s_ptile, G, nct, (T + 127 * (int64_t)G + 127) / 128,
                             (int64_t)blockIdx.x * RW_WARPS + (threadIdx.x >> 5), (int64_t)gridDim.x * RW_WARPS);

}

template <bool GROUPED, bool FOUR_SIX = false>
void launch_rowwise(int64_t T, int64_t H, unsigned grid_cap, size_t smem, cudaStream_t stream, const uint16_t* x,
                    int64_t ldx, uint8_t* q, uint8_t* s, float* s_tok, int G, const int64_t* offs, bool zero_pad = false) {
    if (H / 16 <= 64) {
        const int64_t blocks = (T + RW_WARPS * 2 - 1) / (RW_WARPS * 2);
        nvfp4_rowwise_kernel<GROUPED, 16, FOUR_SIX><<<(unsigned)min64(blocks, grid_cap), RW_WARPS * 32, smem, stream>>>(
            x, T, H, ldx, q, s, s_tok, G, offs, zero_pad);
    } else {
        const int64_t blocks = (T + RW_WARPS - 1) / RW_WARPS;
        nvfp4_rowwise_kernel<GROUPED, 32, FOUR_SIX><<<(unsigned)min64(blocks, grid_cap), RW_WARPS * 32, smem, stream>>>(
            x, T, H, ldx, q, s, s_tok, G, offs, zero_pad);
    }
}

// ------------------------------------------------------------------------------------------------
// Row-wise 1x16 with a per-tensor scale.  With S fixed for the whole tensor the 16-element blocks are
// independent, and a contiguous [T, N] tensor is a flat sequence of them: thread = one block per step
// of a grid-stride loop, the next block's two 16-byte loads issued before the current block is
// quantized.  The reciprocal r of each possible block scale (128 E4M3 codes) is computed once per CTA.
// Block f covers elements 16f .. 16f + 15 (the stochastic-rounding index), row f / (N/16).
// ------------------------------------------------------------------------------------------------
constexpr int FL_THREADS = 256;
constexpr int FL_CTAS_PER_SM = 4;

template <bool SR>
__global__ void __launch_bounds__(FL_THREADS, FL_CTAS_PER_SM)
nvfp4_1x16_flat_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t N, const uint32_t* __restrict__ tensor_amax,
                       float* __restrict__ s_tensor, uint64_t sr_seed, uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
    __shared__ float rtab[128];
    const float S = nvfp4_second_scale(__uint_as_float(*tensor_amax));
    const float rS = nvfp4_fast_rs(S);
    if (threadIdx.x < 128) rtab[threadIdx.x] = nvfp4_block_recip(threadIdx.x, S);
    if (blockIdx.x == 0 && threadIdx.x == 0) *s_tensor = S;
    __syncthreads();

    const int64_t nb = N / 16, total = T * nb, nct = sf_col_tiles(N, 16);
    const int64_t stride = (int64_t)gridDim.x * FL_THREADS;
    const int64_t stride_t = stride / nb, stride_b = stride % nb;
    const bool word_scales = (nb % 4) == 0;        // 4 consecutive blocks from lane 4m share a row
    const uint32_t k0 = (uint32_t)sr_seed, k1 = (uint32_t)(sr_seed >> 32);
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    const int lane = threadIdx.x & 31;

    int64_t f = (int64_t)blockIdx.x * FL_THREADS + threadIdx.x;
    int64_t t = f / nb, b = f % nb;
    uint4 a = make_uint4(0u, 0u, 0u, 0u), c = a;
    if (f < total) { a = __ldcs(xv + 2 * f); c = __ldcs(xv + 2 * f + 1); }
    // warp-uniform trip count (the scale words below use full-warp shuffles)
    for (int64_t fw = f - lane; fw < total; fw += stride) {
        const bool valid = f < total;
        uint4 na = make_uint4(0u, 0u, 0u, 0u), nc = na;
        if (f + stride < total) { na = __ldcs(xv + 2 * (f + stride)); nc = __ldcs(xv + 2 * (f + stride) + 1); }
        uint32_t m2 = 0;
        m2 = absmax_bf16x2(m2, a.x); m2 = absmax_bf16x2(m2, a.y); m2 = absmax_bf16x2(m2, a.z); m2 = absmax_bf16x2(m2, a.w);
        m2 = absmax_bf16x2(m2, c.x); m2 = absmax_bf16x2(m2, c.y); m2 = absmax_bf16x2(m2, c.z); m2 = absmax_bf16x2(m2, c.w);
        const uint32_t bs = nvfp4_block_scale_fast(__uint_as_float(fold_halves(m2) << 16), S, rS);
        const uint2 codes = quant_block16<SR>(a, c, rtab[bs], (uint64_t)f * 16u, k0, k1);
        if (valid) __stcs(reinterpret_cast<uint2*>(q) + f, codes);
        if (word_scales) {
            const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, bs, 1);
            const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, bs, 2);
            const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, bs, 3);
            if (valid && (lane & 3) == 0)
                *reinterpret_cast<uint32_t*>(s + sf_offset(t, b, nct)) = bs | (b1 << 8) | (b2 << 16) | (b3 << 24);
        } else if (valid) {
            s[sf_offset(t, b, nct)] = (uint8_t)bs;
        }
        a = na; c = nc;
        f += stride; t += stride_t; b += stride_b;
        if (b >= nb) { b -= nb; ++t; }
    }
}

// ------------------------------------------------------------------------------------------------
// Column-wise 1x16 along tokens with a per-tensor scale.  CTA tile: 128 tokens x (32 CPT) columns;
// warp w owns tokens [16w, 16w + 16), lane l owns columns [CPT l, CPT l + CPT) (CPT = 8 with
// stochastic rounding, whose Philox block spans 8 columns; 4 otherwise, which halves the registers
// a thread holds and doubles the resident warps).  Each column's 16 codes per warp (8 bytes) are
// staged in shared memory, so that the CTA writes each column's 64 bytes (128 tokens) as whole
// 32-byte sectors; the block scales of a full tile go out as whole 16-byte lines of the scale atoms.
// ------------------------------------------------------------------------------------------------
constexpr int CW_TOK = CW_TILE_TOKENS;
constexpr int CW_THREADS = 256;

// Load a 16 x CPT micro-tile: xw[i] holds row i's CPT BF16 values as CPT / 2 words.
template <int CPT>
__device__ __forceinline__ void load_16(const uint16_t* __restrict__ x, int64_t N, int64_t t0, int64_t n0, bool valid,
                                        uint32_t (&xw)[16][CPT / 2]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        if (CPT == 8) {
            const uint4 v = valid ? __ldcs(reinterpret_cast<const uint4*>(x + (t0 + i) * N + n0)) : make_uint4(0u, 0u, 0u, 0u);
            xw[i][0] = v.x; xw[i][1] = v.y; xw[i][CPT / 2 - 2] = v.z; xw[i][CPT / 2 - 1] = v.w;
        } else {
            const uint2 v = valid ? __ldcs(reinterpret_cast<const uint2*>(x + (t0 + i) * N + n0)) : make_uint2(0u, 0u);
            xw[i][0] = v.x; xw[i][CPT / 2 - 1] = v.y;
        }
    }
}

// The two columns held in word column w of a 16-token micro-tile, transformed in place along the tokens:
// signs applied to the packed BF16 words (a sign flip is exact), butterflies in FP32, x 1/4, and the
// pair packed back to BF16 (RNE), so each word again holds the two columns' values of one token.
template <int NW>
__device__ __forceinline__ void rht16_pair_inplace(uint32_t (&xw)[16][NW], int w, uint32_t signmask) {
    // the two columns as packed FP32 pairs: one instruction per butterfly for both
    uint64_t p[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t v = xw[i][w] ^ (((signmask >> i) & 1u) ? 0x80008000u : 0u);
        p[i] = f2_pack(bf16_lo(v), bf16_hi(v));
    }
    fwht16_unscaled_x2(p);
    const uint64_t q = f2_pack(0.25f, 0.25f);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float lo, hi;
        f2_unpack(f2_mul(p[i], q), lo, hi);
        xw[i][w] = pack_bf16x2(lo, hi);
    }
}

// Tensor amax of the (transformed) input.  With the transform, the maximum is taken over the FP32
// butterfly outputs and scaled by 1/4 and rounded to BF16 once: both steps are monotone in the
// magnitude, so this equals the maximum of the rounded transformed values.
template <bool RHT>
__global__ void __launch_bounds__(CW_THREADS)
colwise_amax_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t N, uint32_t signmask,
                    uint32_t* __restrict__ amax_out) {
    constexpr int CPT = 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)blockIdx.y * CW_TOK + warp * 16;
    const int64_t n0 = (int64_t)blockIdx.x * (32 * CPT) + lane * CPT;
    const bool valid = (t0 < T) && (n0 < N);
    uint32_t xw[16][CPT / 2];
    load_16<CPT>(x, N, t0, n0, valid, xw);
    uint32_t m = 0;
    if (RHT) {
        float mf = 0.0f;
#pragma unroll
        for (int jp = 0; jp < CPT / 2; ++jp) {
            // the two columns of a word transformed together as packed FP32 pairs
            uint64_t v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t w = xw[i][jp] ^ (((signmask >> i) & 1u) ? 0x80008000u : 0u);
                v[i] = f2_pack(bf16_lo(w), bf16_hi(w));
            }
            fwht16_unscaled_x2(v);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float lo, hi;
                f2_unpack(v[i], lo, hi);
                mf = fmaxf(mf, fmaxf(fabsf(lo), fabsf(hi)));
            }
        }
        m = (pack_bf16x2(__fmul_rn(mf, 0.25f), 0.0f) & 0xFFFFu) << 16;
    } else {
        uint32_t m2 = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i)
#pragma unroll
            for (int w = 0; w < CPT / 2; ++w) m2 = absmax_bf16x2(m2, xw[i][w]);
        m = fold_halves(m2) << 16;
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    __shared__ uint32_t wmax[CW_THREADS / 32];
    if (lane == 0) wmax[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = 0;
        for (int i = 0; i < CW_THREADS / 32; ++i) b = max(b, wmax[i]);
        atomicMax(amax_out, b);
    }
}

template <bool RHT, bool SR, int CPT>
__global__ void __launch_bounds__(CW_THREADS, CPT == 8 ? 2 : 3)
colwise_quant_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t N, uint32_t signmask,
                     const uint32_t* __restrict__ tensor_amax, uint64_t sr_seed,
                     uint8_t* __restrict__ q, uint8_t* __restrict__ s, float* __restrict__ s_tensor) {
    static_assert(!SR || CPT == 8, "one Philox block covers 8 columns");
    constexpr int COLS = 32 * CPT;
    __shared__ uint8_t ss[CW_TOK / 16][COLS];                         // block scales: [token block][column]
    // transposed codes: 64 bytes per column, warp w's 8-byte slice in slot w ^ ((column / CPT) & 7), so
    // that the 32 slices one warp stores at a time spread over 8 bank groups
    __shared__ __align__(16) uint8_t qs[COLS * 64];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tb0 = (int64_t)blockIdx.y * CW_TOK;
    const int64_t cb0 = (int64_t)blockIdx.x * COLS;
    const int64_t t0 = tb0 + warp * 16;
    const int64_t n0 = cb0 + lane * CPT;
    const bool valid = (t0 < T) && (n0 < N);

    const float S = nvfp4_second_scale(__uint_as_float(*tensor_amax));
    const float rS = nvfp4_fast_rs(S);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *s_tensor = S;

    uint32_t xw[16][CPT / 2];
    load_16<CPT>(x, N, t0, n0, valid, xw);

    // Phase A, per pair of columns (2 jp, 2 jp + 1), whose values share one BF16 word per token:
    // (transform and re-round in place,) block amax of both columns from the packed words, block
    // scales, reciprocals.
    float rcp[CPT];
#pragma unroll
    for (int jp = 0; jp < CPT / 2; ++jp) {
        if (RHT) rht16_pair_inplace<CPT / 2>(xw, jp, signmask);
        // block maxima of both columns over the 16 packed words (integer pipe: the transform keeps the
        // floating-point pipe busy here)
        uint32_t m2 = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) m2 = absmax_bf16x2_int(m2, xw[i][jp]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = 2 * jp + h;
            const uint32_t bs = nvfp4_block_scale_fast(__uint_as_float((h ? (m2 >> 16) : (m2 & 0xFFFFu)) << 16), S, rS);
            rcp[j] = nvfp4_block_recip(bs, S);
            ss[warp][lane * CPT + j] = (uint8_t)bs;
            if (!SR) {
                float p[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) p[i] = __fmul_rn(h ? bf16_hi(xw[i][jp]) : bf16_lo(xw[i][jp]), rcp[j]);
                // the 16 tokens of column n0 + j: 8 bytes of the transposed output
                *reinterpret_cast<uint2*>(qs + (lane * CPT + j) * 64 + 8 * (warp ^ (lane & 7))) =
                    make_uint2(cvt_e2m1x8(p), cvt_e2m1x8(p + 8));
            }
        }
    }
    if (SR) {
        // Phase B, per row i: one Philox block covers the row's 8 columns (elements t * N + n0 .. + 7)
        const uint32_t k0 = (uint32_t)sr_seed, k1 = (uint32_t)(sr_seed >> 32);
        uint32_t code[CPT][2];
#pragma unroll
        for (int j = 0; j < CPT; ++j) { code[j][0] = 0u; code[j][1] = 0u; }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint64_t blk = ((uint64_t)(t0 + i) * (uint64_t)N + (uint64_t)n0) >> 3;
            const U4 r4 = philox4x32_10((uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u, k0, k1);
            const uint32_t rw[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
            for (int jp = 0; jp < CPT / 2; ++jp) {
                const uint32_t w = xw[i][jp];
                e2m1_sr_pair(__fmul_rn(bf16_lo(w), rcp[2 * jp]), __fmul_rn(bf16_hi(w), rcp[2 * jp + 1]), rw[jp],
                             code[2 * jp][i >> 3], i & 7, code[2 * jp + 1][i >> 3], i & 7);
            }
        }
#pragma unroll
        for (int j = 0; j < CPT; ++j)
            *reinterpret_cast<uint2*>(qs + (lane * CPT + j) * 64 + 8 * (warp ^ (lane & 7))) = make_uint2(code[j][0], code[j][1]);
    }
    __syncthreads();

    const int64_t ntok = min64(CW_TOK, T - tb0);      // multiple of 16
    const int nslot = (int)(ntok / 16);               // 8-byte slices (warps) holding tokens
    // codes: lane 4 c + k writes the 16 bytes of chunk k (tokens tb0 + 32 k .. + 31) of column c
    {
        const bool vec16 = (T / 2) % 16 == 0;
        for (int idx = threadIdx.x; idx < COLS * 4; idx += CW_THREADS) {
            const int c = idx >> 2, k = idx & 3;
            const int64_t n = cb0 + c;
            if (n >= N || 2 * k >= nslot) continue;
            // logical slices 2k, 2k + 1 sit in 16-byte chunk k ^ (m >> 1), swapped when m is odd
            const int m = (c / CPT) & 7;
            uint4 v = *reinterpret_cast<const uint4*>(qs + c * 64 + 16 * (k ^ (m >> 1)));
            if (m & 1) v = make_uint4(v.z, v.w, v.x, v.y);
            uint8_t* dst = q + n * (T / 2) + tb0 / 2 + 16 * k;
            if (vec16 && 2 * k + 1 < nslot) {
                __stcs(reinterpret_cast<uint4*>(dst), v);
            } else {
                __stcs(reinterpret_cast<uint2*>(dst), make_uint2(v.x, v.y));
                if (2 * k + 1 < nslot) __stcs(reinterpret_cast<uint2*>(dst + 8), make_uint2(v.z, v.w));
            }
        }
    }
    const int64_t nct = sf_col_tiles(T, 16);
    if (ntok == CW_TOK && cb0 + COLS <= N) {
        // a full tile's scales are whole 512-byte atoms (128 columns x 4 token blocks): thread i writes
        // line l = i & 31 (columns l, l + 32, l + 64, l + 96 of the atom) of token group (i >> 5) & 1
        for (int idx = threadIdx.x; idx < COLS / 2; idx += CW_THREADS) {
            const int l = idx & 31, grp = (idx >> 5) & 1, an = idx >> 6;
            uint32_t wq[4];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const int col = 128 * an + l + 32 * qq;
                wq[qq] = (uint32_t)ss[4 * grp][col] | ((uint32_t)ss[4 * grp + 1][col] << 8) |
                         ((uint32_t)ss[4 * grp + 2][col] << 16) | ((uint32_t)ss[4 * grp + 3][col] << 24);
            }
            uint8_t* p = s + sf_offset(cb0 + 128 * an, tb0 / 16 + 4 * grp, nct) + 16 * l;
            *reinterpret_cast<uint4*>(p) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
        }
        return;
    }
    // scales: column col gets the 8 block scales of this CTA's 128 tokens (two words of the layout)
    for (int idx = threadIdx.x; idx < COLS * 2; idx += CW_THREADS) {
        const int col = idx >> 1, half = idx & 1;
        const int64_t n = cb0 + col;
        const int64_t kb = tb0 / 16 + half * 4;
        const int nb = (int)min64(4, ntok / 16 - half * 4);
        if (n < N && nb > 0) {
            uint8_t* p = s + sf_offset(n, kb, nct);
            if (nb == 4) {
                *reinterpret_cast<uint32_t*>(p) = (uint32_t)ss[half * 4][col] | ((uint32_t)ss[half * 4 + 1][col] << 8) |
                                                  ((uint32_t)ss[half * 4 + 2][col] << 16) | ((uint32_t)ss[half * 4 + 3][col] << 24);
            } else {
                for (int i = 0; i < nb; ++i) p[i] = ss[half * 4 + i][col];
            }
        }
    }
}

// Plain amax over a BF16 tensor (row-wise per-tensor pass 1).
__global__ void __launch_bounds__(256)
amax_kernel(const uint16_t* __restrict__ x, int64_t n_elems, uint32_t* __restrict__ amax_out) {
    uint32_t m2 = 0;
    const int64_t nvec = n_elems / 8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x) + i);
        m2 = absmax_bf16x2(m2, v.x); m2 = absmax_bf16x2(m2, v.y);
        m2 = absmax_bf16x2(m2, v.z); m2 = absmax_bf16x2(m2, v.w);
    }
    uint32_t m = __reduce_max_sync(0xFFFFFFFFu, fold_halves(m2)) << 16;
    __shared__ uint32_t wmax[8];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = 0;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) b = max(b, wmax[i]);
        atomicMax(amax_out, b);
    }
}

// ------------------------------------------------------------------------------------------------
// Standalone RHT16 along tokens: thread = 16 tokens x 8 columns.
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
rht16_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t N, uint32_t signmask, uint16_t* __restrict__ y) {
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t ncg = N / 8;
    const int64_t t0 = (gid / ncg) * 16, n0 = (gid % ncg) * 8;
    if (t0 >= T) return;
    uint32_t xw[16][4];
    load_16<8>(x, N, t0, n0, true, xw);
#pragma unroll
    for (int w = 0; w < 4; ++w) rht16_pair_inplace<4>(xw, w, signmask);
#pragma unroll
    for (int i = 0; i < 16; ++i)
        __stcs(reinterpret_cast<uint4*>(y + (t0 + i) * N + n0), make_uint4(xw[i][0], xw[i][1], xw[i][2], xw[i][3]));
}

// ------------------------------------------------------------------------------------------------
// 16x16 2D weights.  Pass 1: per-matrix amax.  Pass 2: CTA tile = 64 rows (4 warps x 16) x 128
// columns; lane l reads chunk (l & 15) of rows 2i + (l >> 4); the 16x16 tile amax combines lanes
// l, l^1, l^16 over the 8 iterations.
// ------------------------------------------------------------------------------------------------
constexpr int W2_ROWS = W2D_TILE_ROWS;
constexpr int W2_COLS = 128;

__global__ void __launch_bounds__(256)
matrix_amax_kernel(const uint16_t* __restrict__ w, int64_t per_matrix, uint32_t* __restrict__ amax_out) {
    const int64_t g = blockIdx.y;
    const uint16_t* base = w + g * per_matrix;
    uint32_t m2 = 0;
    const int64_t nvec = per_matrix / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const uint4* vb = reinterpret_cast<const uint4*>(base);
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // four independent 16-byte loads in flight per thread
    for (; i + 3 * stride < nvec; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldg(vb + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            m2 = absmax_bf16x2(m2, v[u].x); m2 = absmax_bf16x2(m2, v[u].y);
            m2 = absmax_bf16x2(m2, v[u].z); m2 = absmax_bf16x2(m2, v[u].w);
        }
    }
    for (; i < nvec; i += stride) {
        const uint4 v = __ldg(vb + i);
        m2 = absmax_bf16x2(m2, v.x); m2 = absmax_bf16x2(m2, v.y);
        m2 = absmax_bf16x2(m2, v.z); m2 = absmax_bf16x2(m2, v.w);
    }
    uint32_t m = __reduce_max_sync(0xFFFFFFFFu, fold_halves(m2)) << 16;
    __shared__ uint32_t wmax[8];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = 0;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) b = max(b, wmax[i]);
        atomicMax(amax_out + g, b);
    }
}

// The work of one lane on its quarter of a 16x16 tile: rows 2 i + rpar (i = 0..7) x the 8 columns of
// xr, the tile's other quarters in lanes l ^ 1, l ^ 16, l ^ 17; rS = nvfp4_fast_rs(S).  Writes this
// lane's row-wise codes (rows o0 + 2 i + rpar at column h), stages its half of the transposed codes
// (8 bytes = the warp's 16 rows of each of 4 columns) at scol_w + 32 c for tile column c, and returns
// the tile's scale code.  All 32 lanes of the warp take part (shuffles); `store` gates the global
// writes only.
template <bool FOUR_SIX>
__device__ __forceinline__ uint32_t w2d_lane_tile(const uint4 (&xr)[8], float S, float rS, int rpar, bool store,
                                                  uint8_t* __restrict__ qrow_g, uint8_t* scol_w,
                                                  int64_t O, int64_t H, int64_t o0, int64_t h, int chunk) {
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        m2 = absmax_bf16x2(m2, xr[i].x); m2 = absmax_bf16x2(m2, xr[i].y);
        m2 = absmax_bf16x2(m2, xr[i].z); m2 = absmax_bf16x2(m2, xr[i].w);
    }
    uint32_t a16 = fold_halves(m2);
    a16 = max(a16, __shfl_xor_sync(0xFFFFFFFFu, a16, 1));
    a16 = max(a16, __shfl_xor_sync(0xFFFFFFFFu, a16, 16));
    // codes of this lane's 8 rows x 8 columns with the tile's scale; with Four-over-Six both candidates
    // (the tile maximum mapped to 6 and to 4) and their largest dequantization errors, combined over the
    // tile's four lanes, decide the scale
    uint32_t codes[8];
    uint32_t bs = 0;
    float err_keep = 0.0f;
#pragma unroll
    for (int k = 0; k < (FOUR_SIX ? 2 : 1); ++k) {
        const uint32_t bsk = nvfp4_block_scale_fast(__uint_as_float(a16 << 16), S, rS, k == 0 ? 6.0f : 4.0f,
                                                    k == 0 ? 1.0f / 6.0f : 0.25f);
        const float r = nvfp4_block_recip(bsk, S);
        uint32_t ck[8];
        float x[64];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x[8 * i + 0] = bf16_lo(xr[i].x); x[8 * i + 1] = bf16_hi(xr[i].x);
            x[8 * i + 2] = bf16_lo(xr[i].y); x[8 * i + 3] = bf16_hi(xr[i].y);
            x[8 * i + 4] = bf16_lo(xr[i].z); x[8 * i + 5] = bf16_hi(xr[i].z);
            x[8 * i + 6] = bf16_lo(xr[i].w); x[8 * i + 7] = bf16_hi(xr[i].w);
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(x[8 * i + j], r);
            ck[i] = cvt_e2m1x8(v);
        }
        if (!FOUR_SIX) {
#pragma unroll
            for (int i = 0; i < 8; ++i) codes[i] = ck[i];
            bs = bsk;
        } else {
            float err = nvfp4_max_dq_error(x, ck, 64, bsk, S);
            err = fmaxf(err, __shfl_xor_sync(0xFFFFFFFFu, err, 1));
            err = fmaxf(err, __shfl_xor_sync(0xFFFFFFFFu, err, 16));
            // the four lanes of a tile hold the same combined error, so they agree on the choice
            if (k == 0 || err < err_keep) {
                err_keep = err;
#pragma unroll
                for (int i = 0; i < 8; ++i) codes[i] = ck[i];
                bs = bsk;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int rr = 2 * i + rpar;                     // row within the warp's 16
        if (store) __stcs(reinterpret_cast<uint32_t*>(qrow_g + (o0 + rr) * (H / 2) + h / 2), codes[i]);
    }
    // transposed copy: lanes l (even rows) and l ^ 16 (odd rows) swap code words; the even-row lane
    // then emits columns 0..3 of its chunk and the odd-row lane columns 4..7, each as the 8 bytes
    // (16 rows, two per byte, even row in the low nibble) of that column's slice.  Per row pair i,
    // byte b of ev[i] holds column 2b (even row's nibble low, odd row's high) and byte b of od[i]
    // column 2b + 1; this lane's columns come from bytes p0 = 2 rpar and p0 + 1, gathered over the 8
    // row pairs by byte permutes.
    uint32_t ev[8], od[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, codes[i], 16);
        const uint32_t e = rpar ? other : codes[i];
        const uint32_t o = rpar ? codes[i] : other;
        ev[i] = (e & 0x0F0F0F0Fu) | ((o << 4) & 0xF0F0F0F0u);
        od[i] = ((e >> 4) & 0x0F0F0F0Fu) | (o & 0xF0F0F0F0u);
    }
    const uint32_t sel = rpar ? 0x7362u : 0x5140u;      // bytes p0 of a, p0 of b, p0 + 1 of a, p0 + 1 of b
    uint32_t col[4][2];                                 // [column - 4 rpar][8-byte half]
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int i0 = 4 * half;
        const uint32_t e01 = __byte_perm(ev[i0], ev[i0 + 1], sel), e23 = __byte_perm(ev[i0 + 2], ev[i0 + 3], sel);
        const uint32_t o01 = __byte_perm(od[i0], od[i0 + 1], sel), o23 = __byte_perm(od[i0 + 2], od[i0 + 3], sel);
        col[0][half] = __byte_perm(e01, e23, 0x5410u);
        col[2][half] = __byte_perm(e01, e23, 0x7632u);
        col[1][half] = __byte_perm(o01, o23, 0x5410u);
        col[3][half] = __byte_perm(o01, o23, 0x7632u);
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
        *reinterpret_cast<uint2*>(scol_w + 32 * (chunk * 8 + jj + 4 * rpar)) = make_uint2(col[jj][0], col[jj][1]);
    return bs;
}

// Row-wise scales of the 16 rows o0 .. o0 + 15 of one warp: 8 tile scales each (tile columns from
// h0 / 16), two words per row; lane l writes word (l & 1) of row o0 + (l >> 1).
__device__ __forceinline__ void w2d_row_scales(const uint8_t (&stw)[W2_COLS / 16], uint8_t* __restrict__ s_row_g,
                                               int64_t O, int64_t H, int64_t o0, int64_t h0, int lane) {
    const int64_t nct = sf_col_tiles(H, 16);
    const int rr = lane >> 1, half = lane & 1;
    const int64_t kb = h0 / 16 + half * 4;
    const int nb = (int)min64(4, H / 16 - kb);
    if (o0 < O && nb > 0) {
        uint8_t* p = s_row_g + sf_offset(o0 + rr, kb, nct);
        if (nb == 4) {
            *reinterpret_cast<uint32_t*>(p) = (uint32_t)stw[half * 4] | ((uint32_t)stw[half * 4 + 1] << 8) |
                                              ((uint32_t)stw[half * 4 + 2] << 16) | ((uint32_t)stw[half * 4 + 3] << 24);
        } else {
            for (int i = 0; i < nb; ++i) p[i] = stw[half * 4 + i];
        }
    }
}

// Quantize pass: one 64 x 128 tile per CTA, each lane loading its own 16-byte chunks.
template <bool FOUR_SIX>
__global__ void __launch_bounds__(128)
weight2d_quant_kernel(const uint16_t* __restrict__ w, int64_t O, int64_t H, const uint32_t* __restrict__ amax,
                      uint8_t* __restrict__ q_row, uint8_t* __restrict__ s_row,
                      uint8_t* __restrict__ q_col, uint8_t* __restrict__ s_col, float* __restrict__ s_w) {
    __shared__ uint8_t st[W2_ROWS / 16][W2_COLS / 16];                 // tile scales
    // transposed codes of the CTA's 64 rows for each of its 128 columns (32 bytes per column, the
    // 8-byte slice of warp w at byte 8 w), written out as whole 32-byte runs
    __shared__ __align__(16) uint8_t scol[W2_COLS * 32];
    // matrices in the reverse of the amax pass's order: the first CTAs find the matrices that pass
    // read last still in L2
    const int64_t g = gridDim.z - 1 - blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t o0 = (int64_t)blockIdx.y * W2_ROWS + warp * 16;
    const int64_t h0 = (int64_t)blockIdx.x * W2_COLS;
    const uint16_t* wg = w + g * O * H;
    const float S = nvfp4_second_scale(__uint_as_float(amax[g]));
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) s_w[g] = S;

    const int chunk = lane & 15, rpar = lane >> 4;
    const int64_t h = h0 + chunk * 8;
    const bool valid = (o0 < O) && (h < H);
    uint4 xr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t o = o0 + 2 * i + rpar;
        xr[i] = valid ? __ldcs(reinterpret_cast<const uint4*>(wg + o * H + h)) : make_uint4(0u, 0u, 0u, 0u);
    }
    const uint32_t bs = w2d_lane_tile<FOUR_SIX>(xr, S, nvfp4_fast_rs(S), rpar, valid, q_row + g * O * (H / 2),
                                                scol + 8 * warp, O, H, o0, h, chunk);
    if (lane < 16 && (lane & 1) == 0) st[warp][lane >> 1] = (uint8_t)bs;
    __syncthreads();

    const int64_t ob = (int64_t)blockIdx.y * W2_ROWS;
    const int64_t nrows = min64(W2_ROWS, O - ob);      // multiple of 16
    const bool full = nrows == W2_ROWS && h0 + W2_COLS <= H;
    // transposed codes: thread t writes 16 bytes (rows ob + 32 half .. + 31) of column (t >> 1) + 64 k;
    // lanes 2c and 2c + 1 fill one 32-byte sector
    {
        uint8_t* qc = q_col + g * H * (O / 2);
        const int half = threadIdx.x & 1;
        const int nslot = (int)(nrows / 16);            // 8-byte slices present
        const bool vec16 = (O / 2) % 16 == 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int c = (threadIdx.x >> 1) + 64 * k;
            const int64_t hc = h0 + c;
            if (hc >= H) continue;
            uint8_t* dst = qc + hc * (O / 2) + ob / 2 + 16 * half;
            const uint2 lo = *reinterpret_cast<const uint2*>(scol + 32 * c + 16 * half);
            const uint2 hi = *reinterpret_cast<const uint2*>(scol + 32 * c + 16 * half + 8);
            if (vec16 && 2 * half + 1 < nslot) {
                __stcs(reinterpret_cast<uint4*>(dst), make_uint4(lo.x, lo.y, hi.x, hi.y));
            } else {
                if (2 * half < nslot) __stcs(reinterpret_cast<uint2*>(dst), lo);
                if (2 * half + 1 < nslot) __stcs(reinterpret_cast<uint2*>(dst + 8), hi);
            }
        }
    }
    const int64_t nct_col = sf_col_tiles(O, 16);
    uint8_t* sbase = s_col + g * host_scale_bytes_dev(H, O, 16);
    if (full) {
        // row-wise scales: thread t < 64 writes rows ob + l and ob + l + 32 (l = t & 31) of scale columns
        // h0 / 16 + 4 (t >> 5) .. + 3, 8 adjacent bytes of the scale atom
        if (threadIdx.x < 64) {
            const int l = threadIdx.x & 31, grp = threadIdx.x >> 5;
            const int64_t nct = sf_col_tiles(H, 16);
            auto word = [&](int r) {
                const uint8_t* t4 = &st[r >> 4][4 * grp];
                return (uint32_t)t4[0] | ((uint32_t)t4[1] << 8) | ((uint32_t)t4[2] << 16) | ((uint32_t)t4[3] << 24);
            };
            uint8_t* p = s_row + g * host_scale_bytes_dev(O, H, 16) + sf_offset(ob + l, h0 / 16 + 4 * grp, nct);
            *reinterpret_cast<uint2*>(p) = make_uint2(word(l), word(l + 32));
        } else if (threadIdx.x >= 96) {
            // column-wise scales: the CTA's 128 columns x 4 row tiles are one whole 512-byte scale atom;
            // lane t writes its 16-byte line (columns t, t + 32, t + 64, t + 96)
            const int t = threadIdx.x - 96;
            uint32_t wq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int jt = (t + 32 * q) >> 4;
                wq[q] = (uint32_t)st[0][jt] | ((uint32_t)st[1][jt] << 8) | ((uint32_t)st[2][jt] << 16) | ((uint32_t)st[3][jt] << 24);
            }
            uint8_t* p = sbase + sf_offset(h0, ob / 16, nct_col) + 16 * t;
            *reinterpret_cast<uint4*>(p) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
        }
        return;
    }
    w2d_row_scales(st[warp], s_row + g * host_scale_bytes_dev(O, H, 16), O, H, o0, h0, lane);
    // column-wise scales: row hc, scale columns ob/16 .. +3 (one word when all 4 row tiles exist)
    {
        const int64_t nct = nct_col;
        const int nb = (int)(nrows / 16);
        for (int c = threadIdx.x; c < W2_COLS; c += 128) {
            const int64_t hc = h0 + c;
            if (hc >= H) continue;
            uint8_t* p = sbase + sf_offset(hc, ob / 16, nct);
            const int jt = c >> 4;
            if (nb == 4) {
                *reinterpret_cast<uint32_t*>(p) = (uint32_t)st[0][jt] | ((uint32_t)st[1][jt] << 8) |
                                                  ((uint32_t)st[2][jt] << 16) | ((uint32_t)st[3][jt] << 24);
            } else {
                for (int i = 0; i < nb; ++i) p[i] = st[i][jt];
            }
        }
    }
}

// The quantize pass of the plain (not Four-over-Six) 2D quantizer.
cudaError_t launch_weight2d_quant_pass(const uint16_t* w, int64_t G, int64_t O, int64_t H, const uint32_t* amax,
                                       uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, float* s_w,
                                       cudaStream_t stream) {
    dim3 grid((unsigned)((H + W2_COLS - 1) / W2_COLS), (unsigned)((O + W2_ROWS - 1) / W2_ROWS), (unsigned)G);
    weight2d_quant_kernel<false><<<grid, 128, 0, stream>>>(w, O, H, amax, q_row, s_row, q_col, s_col, s_w);
    return cudaGetLastError();
}

}  // namespace

// ------------------------------------------------------------------------------------------------
// launchers
// ------------------------------------------------------------------------------------------------
cudaError_t launch_nvfp4_per_token(const uint16_t* x, int64_t T, int64_t H, int64_t ldx, uint8_t* q, uint8_t* s,
                                   float* s_tok, int G, const int64_t* group_offsets, int num_sms, cudaStream_t stream,
                                   bool four_six) {
    // grouped layout: the padding rows between groups and the unused tail are zeroed by the kernel when
    // the scale columns fill whole words; otherwise the whole layout is cleared first
    const bool kernel_pads = G > 0 && ((H / 16) % 4) == 0;
    if (G > 0 && !kernel_pads) {
        cudaError_t e = cudaMemsetAsync(s, 0, (size_t)host_scale_bytes(T + 127 * (int64_t)G, H, 16), stream);
        if (e != cudaSuccess) return e;
    } else if (G == 0 && ((T % 128) != 0 || ((H / 16) % 4) != 0)) {
        cudaError_t e = cudaMemsetAsync(s, 0, (size_t)host_scale_bytes(T, H, 16), stream);
        if (e != cudaSuccess) return e;
    }
    const unsigned cap = (unsigned)num_sms * 16;
    if (G > 0 && four_six)
        launch_rowwise<true, true>(T, H, cap, (size_t)12 * (G + 1) + 128, stream, x, ldx, q, s, s_tok, G, group_offsets,
                                   kernel_pads);
    else if (G > 0)
        launch_rowwise<true>(T, H, cap, (size_t)12 * (G + 1) + 128, stream, x, ldx, q, s, s_tok, G, group_offsets,
                             kernel_pads);
    else if (four_six)
        launch_rowwise<false, true>(T, H, cap, 0, stream, x, ldx, q, s, s_tok, 0, nullptr);
    else
        launch_rowwise<false>(T, H, cap, 0, stream, x, ldx, q, s, s_tok, 0, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4_1x16(const uint16_t* x, int64_t T, int64_t N, bool colwise, bool rht, uint64_t rht_seed,
                              bool sr, uint64_t sr_seed, uint8_t* q, uint8_t* s, float* s_tensor, uint32_t* ws,
                              int num_sms, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
    const int64_t srows = colwise ? N : T, sk = colwise ? T : N;
    if ((srows % 128) != 0 || ((sk / 16) % 4) != 0) {
        e = cudaMemsetAsync(s, 0, (size_t)host_scale_bytes(srows, sk, 16), stream);
        if (e != cudaSuccess) return e;
    }
    if (colwise) {
        const uint32_t mask = rht ? host_rht_sign_mask(rht_seed) : 0u;
        const unsigned gt = (unsigned)((T + CW_TOK - 1) / CW_TOK);
        const dim3 grid4((unsigned)((N + 127) / 128), gt), grid8((unsigned)((N + 255) / 256), gt);
        if (rht) colwise_amax_kernel<true><<<grid4, CW_THREADS, 0, stream>>>(x, T, N, mask, ws);
        else colwise_amax_kernel<false><<<grid4, CW_THREADS, 0, stream>>>(x, T, N, mask, ws);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (rht && sr) colwise_quant_kernel<true, true, 8><<<grid8, CW_THREADS, 0, stream>>>(x, T, N, mask, ws, sr_seed, q, s, s_tensor);
        else if (rht) colwise_quant_kernel<true, false, 4><<<grid4, CW_THREADS, 0, stream>>>(x, T, N, mask, ws, sr_seed, q, s, s_tensor);
        else if (sr) colwise_quant_kernel<false, true, 8><<<grid8, CW_THREADS, 0, stream>>>(x, T, N, mask, ws, sr_seed, q, s, s_tensor);
        else colwise_quant_kernel<false, false, 4><<<grid4, CW_THREADS, 0, stream>>>(x, T, N, mask, ws, sr_seed, q, s, s_tensor);
    } else {
        amax_kernel<<<num_sms * 4, 256, 0, stream>>>(x, T * N, ws);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int64_t blocks = T * (N / 16);
        const unsigned grid = (unsigned)max64(1, min64((blocks + FL_THREADS - 1) / FL_THREADS, (int64_t)num_sms * FL_CTAS_PER_SM));
        if (sr) nvfp4_1x16_flat_kernel<true><<<grid, FL_THREADS, 0, stream>>>(x, T, N, ws, s_tensor, sr_seed, q, s);
        else nvfp4_1x16_flat_kernel<false><<<grid, FL_THREADS, 0, stream>>>(x, T, N, ws, s_tensor, sr_seed, q, s);
    }
    return cudaGetLastError();
}

cudaError_t launch_rht16(const uint16_t* x, int64_t T, int64_t N, uint64_t seed, uint16_t* y, cudaStream_t stream) {
    const int64_t threads = (T / 16) * (N / 8);
    const unsigned grid = (unsigned)((threads + 255) / 256);
    rht16_kernel<<<grid, 256, 0, stream>>>(x, T, N, host_rht_sign_mask(seed), y);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4_weight_2d_given_amax(const uint16_t* w, int64_t G, int64_t O, int64_t H, uint8_t* q_row,
                                              uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, float* s_w,
                                              const uint32_t* amax, cudaStream_t stream) {
    if ((O % 128) != 0 || ((H / 16) % 4) != 0) {
        cudaError_t e = cudaMemsetAsync(s_row, 0, (size_t)(host_scale_bytes(O, H, 16) * G), stream);
        if (e != cudaSuccess) return e;
    }
    if ((H % 128) != 0 || ((O / 16) % 4) != 0) {
        cudaError_t e = cudaMemsetAsync(s_col, 0, (size_t)(host_scale_bytes(H, O, 16) * G), stream);
        if (e != cudaSuccess) return e;
    }
    return launch_weight2d_quant_pass(w, G, O, H, amax, q_row, s_row, q_col, s_col, s_w, stream);
}

cudaError_t launch_nvfp4_weight_2d(const uint16_t* w, int64_t G, int64_t O, int64_t H, uint8_t* q_row, uint8_t* s_row,
                                   uint8_t* q_col, uint8_t* s_col, float* s_w, uint32_t* ws, int num_sms,
                                   cudaStream_t stream, bool four_six) {
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(uint32_t) * (size_t)G, stream);
    if (e != cudaSuccess) return e;
    if ((O % 128) != 0 || ((H / 16) % 4) != 0) {
        e = cudaMemsetAsync(s_row, 0, (size_t)(host_scale_bytes(O, H, 16) * G), stream);
        if (e != cudaSuccess) return e;
    }
    if ((H % 128) != 0 || ((O / 16) % 4) != 0) {
        e = cudaMemsetAsync(s_col, 0, (size_t)(host_scale_bytes(H, O, 16) * G), stream);
        if (e != cudaSuccess) return e;
    }
    const int64_t per = O * H;
    int64_t bx = (per / 8 + 255) / 256;
    const int64_t cap = max64(1, (int64_t)num_sms * 8 / max64(G, 1));
    if (bx > cap) bx = cap;
    matrix_amax_kernel<<<dim3((unsigned)bx, (unsigned)G), 256, 0, stream>>>(w, per, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (!four_six) return launch_weight2d_quant_pass(w, G, O, H, ws, q_row, s_row, q_col, s_col, s_w, stream);
    dim3 grid((unsigned)((H + W2_COLS - 1) / W2_COLS), (unsigned)((O + W2_ROWS - 1) / W2_ROWS), (unsigned)G);
    weight2d_quant_kernel<true><<<grid, 128, 0, stream>>>(w, O, H, ws, q_row, s_row, q_col, s_col, s_w);
    return cudaGetLastError();
}

}  // namespace mxk
