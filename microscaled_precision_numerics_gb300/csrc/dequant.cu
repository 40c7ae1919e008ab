// dequant.cu -- dequantize to BF16 and the byte-mismatch counter.
//
// NVFP4 RL page, "dequantized backward": the backward GEMMs use BF16 operands rebuilt from the exact
// low-precision forward values, y = x * DQ(Q(w_bf16)).
//   MXFP8: y = BF16 RNE of val(q) * 2^(s - 127)        (the FP32 product is exact)
//   NVFP4: y = BF16 RNE of fp32(val(q) * val(bs)) * S  (the first product is exact)
// E2E page abstract / Table 11: the synchronized weights must equal the learner's bytes; the
// mismatch counter is the device-side byte comparison.
#include "mx_internal.h"

namespace mxk {

namespace {

// MXFP8: thread = 16 codes (one uint4) -> 16 BF16 (two uint4).
__global__ void __launch_bounds__(256)
dequant_mxfp8_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t R, int64_t K,
                     uint16_t* __restrict__ y) {
    const int64_t per_row = K / 16;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= R * per_row) return;
    const int64_t r = gid / per_row, k0 = (gid % per_row) * 16;
    const uint32_t sc = __ldg(s + sf_offset(r, k0 / 32, sf_col_tiles(K, 32)));
    // 2^(sc - 127) as FP32; sc = 0 gives the subnormal 2^-127
    const float f = sc == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(sc << 23);
    const uint4 c = __ldcs(reinterpret_cast<const uint4*>(q + r * K + k0));
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a0 = __fmul_rn(e4m3_to_f32(cw[i] & 0xFFu), f);
        const float a1 = __fmul_rn(e4m3_to_f32((cw[i] >> 8) & 0xFFu), f);
        const float a2 = __fmul_rn(e4m3_to_f32((cw[i] >> 16) & 0xFFu), f);
        const float a3 = __fmul_rn(e4m3_to_f32(cw[i] >> 24), f);
        out[2 * i] = pack_bf16x2(a0, a1);
        out[2 * i + 1] = pack_bf16x2(a2, a3);
    }
    uint4* dst = reinterpret_cast<uint4*>(y + r * K + k0);
    __stcs(dst, make_uint4(out[0], out[1], out[2], out[3]));
    __stcs(dst + 1, make_uint4(out[4], out[5], out[6], out[7]));
}

// NVFP4: thread = one 16-block (8 code bytes) -> 16 BF16.
__global__ void __launch_bounds__(256)
dequant_nvfp4_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, const float* __restrict__ s2,
                     int64_t rows_per_scale, int64_t R, int64_t K, uint16_t* __restrict__ y) {
    const int64_t per_row_blk = K / 16;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= R * per_row_blk) return;
    const int64_t r = gid / per_row_blk, b = gid % per_row_blk;
    const float S = rows_per_scale > 0 ? __ldg(s2 + r / rows_per_scale) : __ldg(s2);
    const float bs = e4m3_to_f32(__ldg(s + sf_offset(r, b, sf_col_tiles(K, 16))));
    const uint2 c = __ldcs(reinterpret_cast<const uint2*>(q + r * (K / 2) + b * 8));
    const uint32_t cw[2] = {c.x, c.y};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t h2 = e2m1x2_to_f16x2((cw[i] >> (8 * j)) & 0xFFu);
            const float v0 = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
            const float v1 = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
            out[4 * i + j] = pack_bf16x2(__fmul_rn(__fmul_rn(v0, bs), S), __fmul_rn(__fmul_rn(v1, bs), S));
        }
    }
    uint4* dst = reinterpret_cast<uint4*>(y + r * K + b * 16);
    __stcs(dst, make_uint4(out[0], out[1], out[2], out[3]));
    __stcs(dst + 1, make_uint4(out[4], out[5], out[6], out[7]));
}

// The same for groups of `group_rows` rows sharing one second-level scale, also writing each group's
// max |y| (BF16 bits << 16).  Grid (WPG-warp slices, groups): warp w of group g walks a contiguous slice of
// the group's 16-blocks, lanes on consecutive blocks, and ends with one atomic max, so a group's word
// takes a few dozen atomics rather than one per warp of blocks.
__global__ void __launch_bounds__(256)
dequant_nvfp4_amax_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, const float* __restrict__ s2,
                          int64_t group_rows, int64_t K, uint16_t* __restrict__ y, uint32_t* __restrict__ amax) {
    const int64_t g = blockIdx.y;
    const int64_t per_row_blk = K / 16;
    const int64_t nblk = group_rows * per_row_blk;                   // 16-blocks of the group
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t slice = (nblk + nwarps - 1) / nwarps;
    const int64_t b0 = wid * slice, b1 = min64(nblk, b0 + slice);
    const float S = __ldg(s2 + g);
    const int64_t nct = sf_col_tiles(K, 16);
    uint32_t m2 = 0;
    constexpr int U = 4;                                             // blocks in flight per lane
    for (int64_t gb0 = b0 + (threadIdx.x & 31); gb0 < b1; gb0 += 32 * U) {
        uint2 c[U];
        uint32_t sc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t gb = gb0 + 32 * u;
            c[u] = make_uint2(0u, 0u);
            sc[u] = 0u;
            if (gb < b1) {
                const int64_t r = g * group_rows + gb / per_row_blk, b = gb % per_row_blk;
                sc[u] = __ldg(s + sf_offset(r, b, nct));
                c[u] = __ldcs(reinterpret_cast<const uint2*>(q + r * (K / 2) + b * 8));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t gb = gb0 + 32 * u;
            if (gb >= b1) break;
            const int64_t r = g * group_rows + gb / per_row_blk, b = gb % per_row_blk;
            const float bs = e4m3_to_f32(sc[u]);
            const uint32_t cw[2] = {c[u].x, c[u].y};
            uint32_t out[8];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t h2 = e2m1x2_to_f16x2((cw[i] >> (8 * j)) & 0xFFu);
                    const float v0 = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
                    const float v1 = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
                    out[4 * i + j] = pack_bf16x2(__fmul_rn(__fmul_rn(v0, bs), S), __fmul_rn(__fmul_rn(v1, bs), S));
                    m2 = absmax_bf16x2(m2, out[4 * i + j]);
                }
            }
            uint4* dst = reinterpret_cast<uint4*>(y + r * K + b * 16);
            __stcs(dst, make_uint4(out[0], out[1], out[2], out[3]));
            __stcs(dst + 1, make_uint4(out[4], out[5], out[6], out[7]));
        }
    }
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, fold_halves(m2));
    if ((threadIdx.x & 31) == 0 && b0 < b1) atomicMax(amax + g, m << 16);
}

__global__ void __launch_bounds__(256)
mismatch_kernel(const uint8_t* __restrict__ x, const uint8_t* __restrict__ y, int64_t nbytes,
                unsigned long long* __restrict__ count) {
    unsigned long long local = 0;
    const int64_t nvec = nbytes / 16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        const uint4 a = __ldcs(reinterpret_cast<const uint4*>(x) + i);
        const uint4 b = __ldcs(reinterpret_cast<const uint4*>(y) + i);
        // __vcmpne4 gives 0xFF per differing byte
        local += __popc(__vcmpne4(a.x, b.x)) + __popc(__vcmpne4(a.y, b.y)) +
                 __popc(__vcmpne4(a.z, b.z)) + __popc(__vcmpne4(a.w, b.w));
    }
    local /= 8;
    for (int64_t i = nvec * 16 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nbytes; i += stride)
        local += (x[i] != y[i]) ? 1ull : 0ull;
    for (int o = 16; o > 0; o >>= 1) local += __shfl_down_sync(0xFFFFFFFFu, local, o);
    __shared__ unsigned long long part[8];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = local;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long t = 0;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += part[i];
        if (t) atomicAdd(count, t);
    }
}

}  // namespace

cudaError_t launch_dequant(int fmt, const uint8_t* q, const uint8_t* s, const float* s2, int64_t rows_per_scale,
                           int64_t R, int64_t K, uint16_t* y, cudaStream_t stream) {
    if (fmt == 0) {
        const int64_t threads = R * (K / 16);
        dequant_mxfp8_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(q, s, R, K, y);
    } else {
        const int64_t threads = R * (K / 16);
        dequant_nvfp4_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(q, s, s2, rows_per_scale, R, K, y);
    }
    return cudaGetLastError();
}

cudaError_t launch_dequant_nvfp4_amax(const uint8_t* q, const uint8_t* s, const float* s2, int64_t group_rows, int64_t R,
                                      int64_t K, uint16_t* y, uint32_t* amax, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint32_t) * (size_t)(R / group_rows), stream);
    if (e != cudaSuccess) return e;
    // about 32 CTAs of 8 warps per SM in all (queued, not resident), split evenly over the groups
    const int64_t G = R / group_rows;
    if (G > 65535) return cudaErrorInvalidValue;                     // one grid row per group
    const int64_t per_group = max64(1, (int64_t)device_sm_count() * 32 / G);
    const int64_t need = (group_rows * (K / 16) + 255) / 256;       // no more CTAs than 16-blocks / 256
    dequant_nvfp4_amax_kernel<<<dim3((unsigned)min64(per_group, need), (unsigned)G), 256, 0, stream>>>(q, s, s2, group_rows,
                                                                                                     K, y, amax);
    return cudaGetLastError();
}

cudaError_t launch_mismatch(const uint8_t* x, const uint8_t* y, int64_t nbytes, unsigned long long* count,
                            int num_sms, cudaStream_t stream) {
    int64_t blocks = (nbytes / 16 + 255) / 256;
    blocks = max64(1, min64(blocks, (int64_t)num_sms * 8));
    mismatch_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, y, nbytes, count);
    return cudaGetLastError();
}

}  // namespace mxk
