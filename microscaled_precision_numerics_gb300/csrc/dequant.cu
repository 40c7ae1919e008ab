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

// A thread's 16 BF16 outputs (32 bytes): one 256-bit store when the address is 32-byte aligned (every
// output row starts on a 32-byte boundary when K % 16 == 0 and y is), so that a warp's store fills
// 1 KB of whole lines in one instruction; two 16-byte stores otherwise.
__device__ __forceinline__ void store_bf16x16(uint16_t* dst, const uint32_t (&out)[8]) {
    if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
        asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                     :: "l"(dst), "r"(out[0]), "r"(out[1]), "r"(out[2]), "r"(out[3]), "r"(out[4]), "r"(out[5]),
                        "r"(out[6]), "r"(out[7]) : "memory");
    } else {
        uint4* d = reinterpret_cast<uint4*>(dst);
        __stcs(d, make_uint4(out[0], out[1], out[2], out[3]));
        __stcs(d + 1, make_uint4(out[4], out[5], out[6], out[7]));
    }
}

// The E4M3 block scale in both halves of an FP16 pair (exact: E4M3 values are FP16 values).
__device__ __forceinline__ uint32_t e4m3_to_f16x2_pair(uint32_t code) {
    uint32_t h2;
    asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h2) : "r"((code & 0xFFu) * 0x101u));
    return h2;
}

// value(q) * value(bs) for two codes: the product has at most 6 significant bits and lies in
// [2^-10, 2688] (or is zero), so one packed FP16 multiply gives it exactly, and widening to FP32 gives
// the same two FP32 values as the product taken in FP32.
__device__ __forceinline__ void nvfp4_pair_value(uint32_t q2, uint32_t bs2, float& v0, float& v1) {
    uint32_t p2;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p2) : "r"(q2), "r"(bs2));
    v0 = __half2float(__ushort_as_half((unsigned short)(p2 & 0xFFFFu)));
    v1 = __half2float(__ushort_as_half((unsigned short)(p2 >> 16)));
}

// n / d for the thread-index splits: with 32-bit indices by multiply-high (dv = make_divu32(d); a
// division instruction sequence costs as much as a third of a dequantize thread's work), with 64-bit
// ones plainly.
template <typename Idx>
__device__ __forceinline__ Idx idx_div(Idx n, Idx d, DivU32 dv) {
    if constexpr (sizeof(Idx) == 4) return (Idx)divu32((uint32_t)n, dv);
    else return n / d;
}

// MXFP8: thread = 16 codes (one uint4) -> 16 BF16 (two uint4).  Idx is the type of the thread index and
// of its split into (row, column): 32-bit whenever the tensor has fewer than 2^32 such threads, since a
// 64-bit division costs several times the rest of the thread's work.
template <typename Idx>
__global__ void __launch_bounds__(256)
dequant_mxfp8_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t R, int64_t K,
                     uint16_t* __restrict__ y, DivU32 dv_row) {
    const Idx per_row = (Idx)(K / 16);
    const Idx gid = (Idx)blockIdx.x * (Idx)blockDim.x + (Idx)threadIdx.x;
    if ((int64_t)gid >= R * (int64_t)per_row) return;
    const Idx r_ = idx_div<Idx>(gid, per_row, dv_row);
    const int64_t r = (int64_t)r_, k0 = (int64_t)(gid - r_ * per_row) * 16;
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
    store_bf16x16(y + r * K + k0, out);
}

// NVFP4: thread = one 16-block (8 code bytes) -> 16 BF16 (Idx as above).
template <typename Idx>
__global__ void __launch_bounds__(256)
dequant_nvfp4_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, const float* __restrict__ s2,
                     int64_t rows_per_scale, int64_t R, int64_t K, uint16_t* __restrict__ y, DivU32 dv_row,
                     DivU32 dv_scale) {
    const Idx per_row_blk = (Idx)(K / 16);
    const Idx gid = (Idx)blockIdx.x * (Idx)blockDim.x + (Idx)threadIdx.x;
    if ((int64_t)gid >= R * (int64_t)per_row_blk) return;
    const Idx r_ = idx_div<Idx>(gid, per_row_blk, dv_row);
    const int64_t r = (int64_t)r_, b = (int64_t)(gid - r_ * per_row_blk);
    const float S = rows_per_scale > 0 ? __ldg(s2 + (int64_t)idx_div<Idx>(r_, (Idx)rows_per_scale, dv_scale)) : __ldg(s2);
    const uint32_t bs2 = e4m3_to_f16x2_pair(__ldg(s + sf_offset(r, b, sf_col_tiles(K, 16))));
    const uint2 c = __ldcs(reinterpret_cast<const uint2*>(q + r * (K / 2) + b * 8));
    const uint32_t cw[2] = {c.x, c.y};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float v0, v1;
            nvfp4_pair_value(e2m1x2_to_f16x2((cw[i] >> (8 * j)) & 0xFFu), bs2, v0, v1);
            out[4 * i + j] = pack_bf16x2(__fmul_rn(v0, S), __fmul_rn(v1, S));
        }
    }
    store_bf16x16(y + r * K + b * 16, out);
}

// The same for groups of `group_rows` rows sharing one second-level scale, also writing each group's
// max |y| (BF16 bits << 16).  One 16-block per thread as above; the maxima gather per warp and then per
// CTA (its warps' groups run in order), so a CTA inside one group makes one atomic.  A warp whose lanes
// straddle two groups leaves its maxima to per-lane atomics.
template <typename Idx>
__global__ void __launch_bounds__(256)
dequant_nvfp4_amax_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, const float* __restrict__ s2,
                          int64_t group_rows, int64_t R, int64_t K, uint16_t* __restrict__ y,
                          uint32_t* __restrict__ amax, DivU32 dv_row, DivU32 dv_group) {
    __shared__ uint32_t w_max[8];
    __shared__ int64_t w_grp[8];                                     // -1: nothing left for the CTA to add
    const Idx per_row_blk = (Idx)(K / 16);
    const Idx gid = (Idx)blockIdx.x * (Idx)blockDim.x + (Idx)threadIdx.x;
    // valid threads are a prefix of the grid, so lane 0 of a warp with any valid lane is valid
    const bool valid = (int64_t)gid < R * (int64_t)per_row_blk;
    uint32_t m = 0;
    int64_t g = 0;
    if (valid) {
        const Idx r_ = idx_div<Idx>(gid, per_row_blk, dv_row);
        const int64_t r = (int64_t)r_, b = (int64_t)(gid - r_ * per_row_blk);
        g = (int64_t)idx_div<Idx>(r_, (Idx)group_rows, dv_group);
        const float S = __ldg(s2 + g);
        const uint32_t bs2 = e4m3_to_f16x2_pair(__ldg(s + sf_offset(r, b, sf_col_tiles(K, 16))));
        const uint2 c = __ldcs(reinterpret_cast<const uint2*>(q + r * (K / 2) + b * 8));
        const uint32_t cw[2] = {c.x, c.y};
        uint32_t out[8], m2 = 0;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float v0, v1;
                nvfp4_pair_value(e2m1x2_to_f16x2((cw[i] >> (8 * j)) & 0xFFu), bs2, v0, v1);
                out[4 * i + j] = pack_bf16x2(__fmul_rn(v0, S), __fmul_rn(v1, S));
                m2 = absmax_bf16x2(m2, out[4 * i + j]);
            }
        }
        m = fold_halves(m2);
        store_bf16x16(y + r * K + b * 16, out);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t g0 = __shfl_sync(0xFFFFFFFFu, g, 0);
    const bool one_group = __all_sync(0xFFFFFFFFu, !valid || g == g0);
    const uint32_t mw = __reduce_max_sync(0xFFFFFFFFu, m);
    if (!one_group && valid && m != 0) atomicMax(amax + g, m << 16);
    if (lane == 0) {
        w_max[warp] = mw;
        w_grp[warp] = (one_group && valid) ? g0 : -1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // runs of warps in one group: one atomic per run
        int64_t gc = -1;
        uint32_t mc = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
            if (w_grp[w] < 0) continue;
            if (w_grp[w] != gc) {
                if (gc >= 0 && mc != 0) atomicMax(amax + gc, mc << 16);
                gc = w_grp[w];
                mc = 0;
            }
            mc = max(mc, w_max[w]);
        }
        if (gc >= 0 && mc != 0) atomicMax(amax + gc, mc << 16);
    }
}

__global__ void __launch_bounds__(256)
mismatch_kernel(const uint8_t* __restrict__ x, const uint8_t* __restrict__ y, int64_t nbytes,
                unsigned long long* __restrict__ count) {
    unsigned long long local = 0;
    const int64_t nvec = nbytes / 16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // MU vector pairs in flight per thread before the first compare
    constexpr int MU = 4;
    for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < nvec; i0 += MU * stride) {
        uint4 a[MU], b[MU];
#pragma unroll
        for (int u = 0; u < MU; ++u) {
            const int64_t i = i0 + u * stride;
            a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
            if (i < nvec) {
                a[u] = __ldcs(reinterpret_cast<const uint4*>(x) + i);
                b[u] = __ldcs(reinterpret_cast<const uint4*>(y) + i);
            }
        }
#pragma unroll
        for (int u = 0; u < MU; ++u) {
            // __vcmpne4 gives 0xFF per differing byte
            local += __popc(__vcmpne4(a[u].x, b[u].x)) + __popc(__vcmpne4(a[u].y, b[u].y)) +
                     __popc(__vcmpne4(a[u].z, b[u].z)) + __popc(__vcmpne4(a[u].w, b[u].w));
        }
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
    const int64_t threads = R * (K / 16);
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    const bool idx32 = threads + 256 <= (int64_t)UINT32_MAX;       // every thread index fits 32 bits
    const DivU32 dv_row = make_divu32((uint64_t)(K / 16));
    const DivU32 dv_scale = make_divu32(rows_per_scale > 0 ? (uint64_t)rows_per_scale : 1u);
    if (fmt == 0) {
        if (idx32) dequant_mxfp8_kernel<uint32_t><<<blocks, 256, 0, stream>>>(q, s, R, K, y, dv_row);
        else dequant_mxfp8_kernel<int64_t><<<blocks, 256, 0, stream>>>(q, s, R, K, y, dv_row);
    } else {
        if (idx32) dequant_nvfp4_kernel<uint32_t><<<blocks, 256, 0, stream>>>(q, s, s2, rows_per_scale, R, K, y, dv_row, dv_scale);
        else dequant_nvfp4_kernel<int64_t><<<blocks, 256, 0, stream>>>(q, s, s2, rows_per_scale, R, K, y, dv_row, dv_scale);
    }
    return cudaGetLastError();
}

cudaError_t launch_dequant_nvfp4_amax(const uint8_t* q, const uint8_t* s, const float* s2, int64_t group_rows, int64_t R,
                                      int64_t K, uint16_t* y, uint32_t* amax, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint32_t) * (size_t)(R / group_rows), stream);
    if (e != cudaSuccess) return e;
    const int64_t threads = R * (K / 16);
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    const DivU32 dv_row = make_divu32((uint64_t)(K / 16)), dv_group = make_divu32((uint64_t)group_rows);
    if (threads + 256 <= (int64_t)UINT32_MAX)
        dequant_nvfp4_amax_kernel<uint32_t><<<blocks, 256, 0, stream>>>(q, s, s2, group_rows, R, K, y, amax, dv_row, dv_group);
    else
        dequant_nvfp4_amax_kernel<int64_t><<<blocks, 256, 0, stream>>>(q, s, s2, group_rows, R, K, y, amax, dv_row, dv_group);
    return cudaGetLastError();
}

cudaError_t launch_mismatch(const uint8_t* x, const uint8_t* y, int64_t nbytes, unsigned long long* count,
                            int num_sms, cudaStream_t stream) {
    // one wave: 40 registers a thread leave room for 6 CTAs of 256 threads per SM
    int64_t blocks = (nbytes / 16 + 255) / 256;
    blocks = max64(1, min64(blocks, (int64_t)num_sms * 6));
    mismatch_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, y, nbytes, count);
    return cudaGetLastError();
}

}  // namespace mxk
