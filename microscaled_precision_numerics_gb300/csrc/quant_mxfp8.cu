// quant_mxfp8.cu -- MXFP8 (1x32 and 32x1 E4M3 blocks with E8M0 scales) quantizer, row-wise and
// column-wise copies from one read of the BF16 input.
//
// Miles page: MXFP8 = 32 E4M3 values sharing one E8M0 scale; the tensor cores want the blocks along
// the GEMM's reduction dimension, so TransformerEngine makes row-wise and column-wise copies from
// the high-precision input.  E2E page Table 6: the quantizer and a separate scale-rearrangement
// kernel cost 2.2 + 2.6 ms per micro-batch; here one kernel writes both copies with their scales
// already in the GEMM layout.
//
// CTA tile: 128 rows x 128 columns of BF16 (32 KB), brought into shared memory by TMA (128-byte
// swizzle); both passes read it with 16-byte loads and keep the values in registers between amax and
// conversion.
// Scale exponent: e = max(exp_field(amax) - 8, 0) - 127 as an E8M0 byte; the multiply by 2^-e is
// exact in FP32 for every value that can round to a nonzero E4M3 code.
#include "../../include/mxnum.h"
#include "mx_internal.h"
#include "mx_async.cuh"

#include <cstring>

namespace mxk {

namespace {

constexpr int QT_ROWS = 128;
constexpr int QT_COLS = 128;
constexpr int QT_THREADS = 256;

__device__ __forceinline__ uint32_t e8m0_from_amax_bits(uint32_t amax16) {
    const int ef = (int)((amax16 >> 7) & 0xFFu);   // BF16 exponent field (0 for zero/subnormal)
    return (uint32_t)max(ef - 8, 0);                 // clamp e = ef - 127 - 8 at -127
}

// 2^-e for scale byte s (e = s - 127): exponent field 254 - s, always a normal FP32.
__device__ __forceinline__ float inv_scale_from_e8m0(uint32_t s) { return __uint_as_float((254u - s) << 23); }

// Quantize 32 BF16 values held as 16 packed words; writes 32 code bytes into out[8] words.
__device__ __forceinline__ uint32_t mxfp8_block32(const uint32_t w[16], uint32_t out[8], uint32_t& amax16) {
    uint32_t m2 = absmax_bf16x2(w[0], w[1]);
#pragma unroll
    for (int i = 2; i < 16; ++i) m2 = absmax_bf16x2(m2, w[i]);
    amax16 = fold_halves(m2);
    const uint32_t s = e8m0_from_amax_bits(amax16);
    const float f = inv_scale_from_e8m0(s);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        out[i] = cvt_e4m3x4(__fmul_rn(bf16_lo(w[2 * i]), f), __fmul_rn(bf16_hi(w[2 * i]), f),
                            __fmul_rn(bf16_lo(w[2 * i + 1]), f), __fmul_rn(bf16_hi(w[2 * i + 1]), f));
    }
    return s;
}

// Element j (0..7) of a 16-byte chunk of 8 BF16 values.
__device__ __forceinline__ float chunk_elem(const uint4& v, int j) {
    const uint32_t w = (j >> 1) == 0 ? v.x : ((j >> 1) == 1 ? v.y : ((j >> 1) == 2 ? v.z : v.w));
    return (j & 1) ? bf16_hi(w) : bf16_lo(w);
}

__device__ unsigned int g_mx8_status = 0;

constexpr int QT_CONSUMERS = QT_THREADS;               // 8 consumer warps
constexpr int QT_BLOCK = QT_CONSUMERS + 32;            // + 1 producer warp
constexpr int QT_NST = 2;                              // ring stages of one 32 KB tile
constexpr int QT_CTAS_PER_SM = 3;                      // occupancy hides the passes' dependent chains
constexpr int QT_TILE_BYTES = QT_ROWS * QT_COLS * 2;
constexpr int QT_BOX_BYTES = QT_TILE_BYTES / 2;        // 128 rows x 64 columns (128 bytes)

// Up to MX8_MAX_BATCH tensors quantized by one launch: their 128 x 128 tiles are numbered one tensor
// after the other (tile_end = running totals), and each tile is looked up here by its number.
struct alignas(64) Mx8Params {
    CUtensorMap tm[MX8_MAX_BATCH];      // [R, K] BF16 with row pitch ldx, 128 x 64 boxes, 128-byte swizzle
    int64_t R[MX8_MAX_BATCH], K[MX8_MAX_BATCH], tiles_c[MX8_MAX_BATCH], tile_end[MX8_MAX_BATCH];
    uint8_t* q_row[MX8_MAX_BATCH];
    uint8_t* s_row[MX8_MAX_BATCH];
    uint8_t* q_col[MX8_MAX_BATCH];
    uint8_t* s_col[MX8_MAX_BATCH];
    uint32_t* amax;           // optional (one tensor): per-matrix max |x| as BF16 bits << 16
    int64_t matrix_rows;      // rows per matrix for `amax` (a multiple of 128)
    int n;
};

template <typename T>
__device__ __forceinline__ T pick(const T (&a)[MX8_MAX_BATCH], int i) {
    T v = a[0];
#pragma unroll
    for (int j = 1; j < MX8_MAX_BATCH; ++j) v = (i == j) ? a[j] : v;
    return v;
}

// The tensor that tile number t belongs to.
__device__ __forceinline__ int tile_tensor(const Mx8Params& p, int64_t t) {
    int i = 0;
#pragma unroll
    for (int j = 1; j < MX8_MAX_BATCH; ++j) i = (j < p.n && t >= p.tile_end[j - 1]) ? j : i;
    return i;
}

// Byte offset of 16-byte chunk c (0..15 along the 128 columns) of tile row r in a staged tile: two TMA
// boxes of 128 rows x 128 bytes (columns 0..63, 64..127), each with the 128-byte swizzle (chunk index
// XOR row & 7), which keeps both passes' 16-byte shared loads free of bank conflicts.
__device__ __forceinline__ uint32_t qt_off(int r, int c) {
    return (uint32_t)((c >> 3) * QT_BOX_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void named_sync_consumers() { asm volatile("bar.sync 1, %0;" :: "r"(QT_CONSUMERS) : "memory"); }

// Persistent CTAs (three per SM) walk the 128 x 128 tiles; warp 0 streams them through a 2-stage ring
// by TMA, warps 1..8 quantize:
//   row pass:    thread -> (row, pair of 32-column blocks); 8 x 16-byte shared loads
//   column pass: thread -> (8-column chunk, 32-row block, quarter of 8 rows); 8 x 16-byte shared
//                loads; the 32-row amax combines the 4 quarters (lanes l, l^8, l^16, l^24)
template <bool ROW, bool COL, bool GROUPED>
__global__ void __launch_bounds__(QT_BLOCK, QT_CTAS_PER_SM)
mxfp8_quantize_kernel(const __grid_constant__ Mx8Params p, int G, const int64_t* __restrict__ group_offsets,
                      bool zero_pad) {
    using namespace async;
    extern __shared__ uint8_t qsm_raw[];
    uint8_t* qsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsm_raw) + 1023) & ~uintptr_t(1023));
    uint8_t (*colsc)[QT_COLS] = reinterpret_cast<uint8_t (*)[QT_COLS]>(qsm + QT_NST * QT_TILE_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(qsm + QT_NST * QT_TILE_BYTES + 4 * QT_COLS);   // full[3], empty[3]
    int* abort_flag = reinterpret_cast<int*>(bars + 2 * QT_NST);
    __shared__ uint32_t tile_amax[2];                       // per-tile maxima (optional output), by tile parity
    // expert-group tables (grouped row-wise scale layout)
    int64_t* s_off = reinterpret_cast<int64_t*>(qsm + QT_NST * QT_TILE_BYTES + 4 * QT_COLS + 64);
    int* s_ptile = reinterpret_cast<int*>(s_off + (G + 1));
    int* s_warp = s_ptile + (G + 1);
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * QT_NST;
    if (threadIdx.x == 0) {
        for (int st = 0; st < QT_NST; ++st) {
            mbar_init(full0 + 8 * st, 1);
            mbar_init(empty0 + 8 * st, 1);
        }
        *abort_flag = 0;
        tile_amax[0] = tile_amax[1] = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (GROUPED) load_group_tables(group_offsets, G, s_off, s_ptile, s_warp);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles = p.tile_end[p.n - 1];
    if (warp == 0) {
        // ------------------------------- producer -------------------------------
        if (lane < p.n) asm volatile("prefetch.tensormap [%0];" :: "l"(&p.tm[lane]) : "memory");
        uint32_t k = 0;
        for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++k) {
            const uint32_t stage = k % QT_NST, phase = (k / QT_NST) & 1u;
            if (!warp_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, &g_mx8_status)) break;
            if (elect_one()) {
                const int i = tile_tensor(p, t);
                const int64_t lt = t - (i > 0 ? pick(p.tile_end, i - 1) : 0), tc = pick(p.tiles_c, i);
                const int32_t r0 = (int32_t)((lt / tc) * QT_ROWS), c0 = (int32_t)((lt % tc) * QT_COLS);
                const uint32_t dst = smem_u32(qsm + stage * QT_TILE_BYTES);
                mbar_arrive_expect_tx(full0 + 8 * stage, QT_TILE_BYTES);
                tma_load_2d(dst, &p.tm[i], c0, r0, full0 + 8 * stage);
                tma_load_2d(dst + QT_BOX_BYTES, &p.tm[i], c0 + 64, r0, full0 + 8 * stage);
            }
            __syncwarp();
        }
        return;
    }
    const int tid = threadIdx.x - 32, cw = tid >> 5;         // consumer thread / warp
    uint32_t k = 0;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++k) {
        const uint32_t stage = k % QT_NST, phase = (k / QT_NST) & 1u;
        // warp-uniform: the passes below use full-warp shuffles
        const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * stage, phase, abort_flag, &g_mx8_status)) != 0;
        const uint8_t* tile = qsm + stage * QT_TILE_BYTES;
        const int ti = tile_tensor(p, t);
        const int64_t lt = t - (ti > 0 ? pick(p.tile_end, ti - 1) : 0), tiles_c = pick(p.tiles_c, ti);
        const int64_t R = pick(p.R, ti), K = pick(p.K, ti);
        uint8_t* __restrict__ q_row = pick(p.q_row, ti);
        uint8_t* __restrict__ s_row = pick(p.s_row, ti);
        uint8_t* __restrict__ q_col = pick(p.q_col, ti);
        uint8_t* __restrict__ s_col = pick(p.s_col, ti);
        const int64_t r0 = (lt / tiles_c) * QT_ROWS;
        const int64_t c0 = (lt % tiles_c) * QT_COLS;

        if (ROW && ok) {
            // lanes 0..7 take 8 different rows of the same 64-column half
            const int half = (tid >> 3) & 1;
            const int rr = (tid & 7) + 8 * (tid >> 4);
            const int64_t r = r0 + rr;
            uint32_t s2[2], am = 0;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = *reinterpret_cast<const uint4*>(tile + qt_off(rr, half * 8 + b * 4 + i));
                    w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
                }
                uint32_t codes[8], a16;
                s2[b] = mxfp8_block32(w, codes, a16);
                am = max(am, a16);
                const int64_t c = c0 + half * 64 + b * 32;
                if (r < R && c < K) {
                    stcs_32b(q_row + r * K + c, make_uint4(codes[0], codes[1], codes[2], codes[3]),
                             make_uint4(codes[4], codes[5], codes[6], codes[7]));
                }
            }
            if (p.amax != nullptr) {
                // the tile's maximum gathers in shared memory (one global atomic per tile, below)
                am = __reduce_max_sync(0xFFFFFFFFu, am);
                if (lane == 0) atomicMax(&tile_amax[k & 1], am);
            }
            // the row's 4 scales: this thread's two and those of lane + 8 (the other half)
            const uint32_t mine = s2[0] | (s2[1] << 8);
            const uint32_t other = __shfl_down_sync(0xFFFFFFFFu, mine, 8);
            const int64_t srow = GROUPED ? grouped_scale_row(s_off, s_ptile, G, r) : r;
            // (a grouped row stays inside the layout even for offsets that are not non-decreasing)
            if (half == 0 && r < R && srow >= 0 && srow < R + 127 * (int64_t)G) {
                const int64_t nct = sf_col_tiles(K, 32);
                const int nvalid = (int)min64(4, (K - c0) / 32);
                uint8_t* p = s_row + sf_offset(srow, c0 / 32, nct);
                const uint32_t word = mine | (other << 16);
                if (nvalid == 4) *reinterpret_cast<uint32_t*>(p) = word;
                else for (int i = 0; i < nvalid; ++i) p[i] = (uint8_t)(word >> (8 * i));
            }
        }

        if (COL && ok) {
            const int rb = cw >> 1;                          // 32-row block
            const int chunk = (cw & 1) * 8 + (lane & 7);     // 8-column chunk
            const int q = lane >> 3;                         // quarter: rows q*8 .. q*8+7 of the block
            uint4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = *reinterpret_cast<const uint4*>(tile + qt_off(rb * 32 + q * 8 + i, chunk));
            uint32_t m[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
#pragma unroll
            for (int i = 1; i < 8; ++i) {
                m[0] = absmax_bf16x2(m[0], v[i].x); m[1] = absmax_bf16x2(m[1], v[i].y);
                m[2] = absmax_bf16x2(m[2], v[i].z); m[3] = absmax_bf16x2(m[3], v[i].w);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                m[kk] = absmax_bf16x2(m[kk], __shfl_xor_sync(0xFFFFFFFFu, m[kk], 8));
                m[kk] = abs_halves(absmax_bf16x2(m[kk], __shfl_xor_sync(0xFFFFFFFFu, m[kk], 16)));
            }
            const int64_t rbase = r0 + rb * 32;
            const bool rows_ok = rbase < R;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t a16 = (j & 1) ? (m[j >> 1] >> 16) : (m[j >> 1] & 0xFFFFu);
                const uint32_t sc = e8m0_from_amax_bits(a16);
                const float f = inv_scale_from_e8m0(sc);
                const uint32_t lo = cvt_e4m3x4(__fmul_rn(chunk_elem(v[0], j), f), __fmul_rn(chunk_elem(v[1], j), f),
                                               __fmul_rn(chunk_elem(v[2], j), f), __fmul_rn(chunk_elem(v[3], j), f));
                const uint32_t hi = cvt_e4m3x4(__fmul_rn(chunk_elem(v[4], j), f), __fmul_rn(chunk_elem(v[5], j), f),
                                               __fmul_rn(chunk_elem(v[6], j), f), __fmul_rn(chunk_elem(v[7], j), f));
                const int64_t c = c0 + chunk * 8 + j;
                if (rows_ok && c < K)
                    __stcs(reinterpret_cast<uint2*>(q_col + c * R + rbase + q * 8), make_uint2(lo, hi));
                if (q == 0) colsc[rb][chunk * 8 + j] = (uint8_t)sc;
            }
        }
        // both passes have read the stage: hand it back to the producer
        named_sync_consumers();
        if (tid == 0) mbar_arrive(empty0 + 8 * stage);
        if (p.amax != nullptr && tid == 0) {
            // the tile lies in one matrix (128-row tiles, matrices a multiple of 128 rows); this slot is
            // next written two tiles on, after this thread has passed the next tile's barrier
            if (ok && r0 < R) atomicMax(p.amax + r0 / p.matrix_rows, tile_amax[k & 1] << 16);
            tile_amax[k & 1] = 0u;
        }
        if (COL) {
            // one 32-bit word of 4 row-block scales per column (r0 / 32 is a multiple of 4)
            if (ok && tid < QT_COLS) {
                const int64_t cw_ = c0 + tid;
                if (cw_ < K) {
                    const int64_t nct = sf_col_tiles(R, 32);
                    const int nvalid = (int)min64(4, (R - r0) / 32);
                    uint8_t* p = s_col + sf_offset(cw_, r0 / 32, nct);
                    if (nvalid == 4) {
                        *reinterpret_cast<uint32_t*>(p) = (uint32_t)colsc[0][tid] | ((uint32_t)colsc[1][tid] << 8) |
                                                          ((uint32_t)colsc[2][tid] << 16) | ((uint32_t)colsc[3][tid] << 24);
                    } else {
                        for (int i = 0; i < nvalid; ++i) p[i] = colsc[i][tid];
                    }
                }
            }
            named_sync_consumers();   // colsc is rewritten by the next tile
        }
    }
    if (GROUPED && zero_pad)
        zero_grouped_padding(p.s_row[0], s_off, s_ptile, G, sf_col_tiles(p.K[0], 32), (p.R[0] + 127 * (int64_t)G + 127) / 128,
                             (int64_t)blockIdx.x * (QT_CONSUMERS / 32) + cw, (int64_t)gridDim.x * (QT_CONSUMERS / 32));
    if (*abort_flag && tid == 0) {
        // after an expired wait: give loads already issued by this CTA time to land before exit
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {}
    }
}

// Scale padding that the kernel does not write (rows beyond R up to a multiple of 128, scale columns up to
// a multiple of 4; in the grouped layout also the rows between groups) is zeroed first.
static cudaError_t mx8_zero_padding(const Mx8Tensor& t, int G, cudaStream_t stream) {
    // grouped with whole scale words: the kernel zeroes the padding rows between groups and the tail
    if (t.q_row && ((G > 0 && ((t.K / 32) % 4) != 0) || (G == 0 && ((t.R % 128) != 0 || ((t.K / 32) % 4) != 0)))) {
        cudaError_t e = cudaMemsetAsync(t.s_row, 0, (size_t)host_scale_bytes(t.R + 127 * (int64_t)G, t.K, 32), stream);
        if (e != cudaSuccess) return e;
    }
    if (t.q_col && ((t.K % 128) != 0 || ((t.R / 32) % 4) != 0)) {
        cudaError_t e = cudaMemsetAsync(t.s_col, 0, (size_t)host_scale_bytes(t.K, t.R, 32), stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

static cudaError_t launch_mx8(const Mx8Tensor* ts, int n, int G, const int64_t* group_offsets, cudaStream_t stream,
                              uint32_t* amax = nullptr, int64_t matrix_rows = 0) {
    if (n < 1 || n > MX8_MAX_BATCH) return cudaErrorInvalidValue;
    if (amax && (n != 1 || G > 0 || !ts[0].q_row || matrix_rows <= 0 || (matrix_rows % 128) != 0 ||
                 (ts[0].R % matrix_rows) != 0))
        return cudaErrorInvalidValue;
    const bool row = ts[0].q_row != nullptr, col = ts[0].q_col != nullptr;
    Mx8Params p;
    memset(&p, 0, sizeof(p));
    p.n = n;
    int64_t tiles = 0;
    for (int i = 0; i < n; ++i) {
        const Mx8Tensor& t = ts[i];
        if ((t.q_row != nullptr) != row || (t.q_col != nullptr) != col) return cudaErrorInvalidValue;
        if (!encode_tensor_map_2d(&p.tm[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, t.x, (uint64_t)t.K, (uint64_t)t.R,
                                  (uint64_t)(t.ldx * 2), 64, QT_ROWS, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
            return cudaErrorInvalidValue;
        p.R[i] = t.R; p.K[i] = t.K;
        p.tiles_c[i] = (t.K + QT_COLS - 1) / QT_COLS;
        tiles += p.tiles_c[i] * ((t.R + QT_ROWS - 1) / QT_ROWS);
        p.tile_end[i] = tiles;
        p.q_row[i] = t.q_row; p.s_row[i] = t.s_row; p.q_col[i] = t.q_col; p.s_col[i] = t.s_col;
    }
    p.amax = amax;
    p.matrix_rows = matrix_rows;
    // every descriptor is valid: only now enqueue anything
    for (int i = 0; i < n; ++i) {
        cudaError_t e = mx8_zero_padding(ts[i], G, stream);
        if (e != cudaSuccess) return e;
    }
    if (amax) {
        cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint32_t) * (size_t)(ts[0].R / matrix_rows), stream);
        if (e != cudaSuccess) return e;
    }
    const size_t base = (size_t)QT_NST * QT_TILE_BYTES + 4 * QT_COLS + 64 + 1024;
    const size_t smem = base + (G > 0 ? (size_t)12 * (G + 1) + 128 : 0);
    static PerDevice setup;
    int unused = 0;
    const cudaError_t attr_err = per_device_once(setup, unused, [base](int&) -> cudaError_t {
        const int max_smem = (int)(base + 12 * (MX_MAX_GROUPS + 1) + 128);
        const void* ks[] = {(const void*)mxfp8_quantize_kernel<true, true, false>, (const void*)mxfp8_quantize_kernel<true, false, false>,
                            (const void*)mxfp8_quantize_kernel<false, true, false>, (const void*)mxfp8_quantize_kernel<true, false, true>};
        for (const void* kf : ks) {
            const cudaError_t e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    });
    if (attr_err != cudaSuccess) return attr_err;
    const unsigned grid = (unsigned)min64(tiles, (int64_t)device_sm_count() * QT_CTAS_PER_SM);
    if (G > 0)
        mxfp8_quantize_kernel<true, false, true><<<grid, QT_BLOCK, smem, stream>>>(p, G, group_offsets,
                                                                                    ((ts[0].K / 32) % 4) == 0);
    else if (row && col)
        mxfp8_quantize_kernel<true, true, false><<<grid, QT_BLOCK, smem, stream>>>(p, 0, nullptr, false);
    else if (row)
        mxfp8_quantize_kernel<true, false, false><<<grid, QT_BLOCK, smem, stream>>>(p, 0, nullptr, false);
    else
        mxfp8_quantize_kernel<false, true, false><<<grid, QT_BLOCK, smem, stream>>>(p, 0, nullptr, false);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mxfp8_quantize(const uint16_t* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q_row,
                                  uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, int G, const int64_t* group_offsets,
                                  cudaStream_t stream) {
    const Mx8Tensor t{x, R, K, ldx, q_row, s_row, q_col, s_col};
    return launch_mx8(&t, 1, G, group_offsets, stream);
}

cudaError_t launch_mxfp8_quantize_batched(const Mx8Tensor* ts, int n, cudaStream_t stream) {
    return launch_mx8(ts, n, 0, nullptr, stream);
}

cudaError_t launch_mxfp8_quantize_amax(const Mx8Tensor& t, int64_t matrix_rows, uint32_t* amax, cudaStream_t stream) {
    return launch_mx8(&t, 1, 0, nullptr, stream, amax, matrix_rows);
}

uint32_t read_and_clear_mxfp8_status() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_mx8_status, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    cudaMemcpyToSymbol(g_mx8_status, &zero, sizeof(zero));
    return v;
}

uint32_t read_and_clear_mxfp8_status_on(cudaStream_t stream) {
    unsigned int v = 0;
    static const unsigned int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_mx8_status, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_mx8_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return 0xFFFFFFFFu;
    return v;
}

namespace {
// Watchdog self-test of this file's status word: one CTA whose warps wait on a barrier that nothing
// arrives on (the quantizer's ring waits, with the caller's limit); the first to give up sets the
// timeout bit and the abort flag, the others leave on the flag.  No copy is ever issued.
__global__ void __launch_bounds__(288) mx8_watchdog_selftest_kernel(unsigned long long limit_ns) {
    using namespace async;
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_s;
    volatile int* abort_flag = &abort_s;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    warp_wait(smem_u32(&bar), 0, abort_flag, &g_mx8_status, limit_ns);
    __syncthreads();
}
}  // namespace

cudaError_t launch_mxfp8_watchdog_selftest(unsigned long long limit_ns, cudaStream_t stream) {
    mx8_watchdog_selftest_kernel<<<1, 288, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

}  // namespace mxk
