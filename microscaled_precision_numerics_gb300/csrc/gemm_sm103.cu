// gemm_sm103.cu -- block-scaled GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   D[m, n] = BF16( alpha_a[m] * alpha_b[n] * sum_k DQ(A)[m, k] * DQ(B)[n, k] )
//
// Miles page: MXFP8 forward, weight-gradient and data-gradient GEMMs; MaxText page: the three MLP
// GEMMs take NVFP4 inputs and emit BF16; E2E page Table 6: GEMM time per micro-batch.  MXFP8 uses
// tcgen05.mma kind::mxf8f6f4 with one E8M0 scale per 32 (scale_vec::1X); NVFP4 uses kind::mxf4nvf4
// with one E4M3 scale per 16 (scale_vec::4X); the FP32 second-level scales are applied in the
// epilogue.
//
// Structure: persistent clusters of two CTAs (one per SM) over 256 x 256 output tiles (256 x 384 for
// large dense MXFP8 GEMMs).  The even CTA issues the pair MMA (tcgen05.mma.cta_group::2, M = 256):
// each CTA holds 128 rows of A and half of the B rows in its shared memory and 128 accumulator rows
// in its TMEM, so each SM loads half of the B tile.
//   warp 0        (both CTAs) TMA producer: A rows, B half and scale atoms (128-byte swizzle for the
//                 operands) into a 6-stage (MXFP8) / 5-stage (NVFP4) ring; the loads of both CTAs
//                 signal the stage barrier in the even CTA
//   warp 1        TMEM allocation for the pair; in the even CTA one elected lane copies each stage's
//                 scale atoms into the TMEM of both CTAs (tcgen05.cp.cta_group::2: each CTA's own
//                 atoms into its own TMEM) and issues the stage's MMAs, which the tensor pipe runs in
//                 issue order; its commits arrive on the barriers of both CTAs
//   warps 2..9    (both CTAs) epilogue, two warps per TMEM lane quadrant (one per column half):
//                 load the row's FP32 scales before the accumulator is ready, tcgen05.ld the
//                 accumulator, scale, round to BF16, hand TMEM back (arriving in the even CTA), then
//                 stage 32-row x 16-column BF16 chunks in swizzled shared memory and write them with
//                 TMA tensor stores (the map clips ragged edges)
// The producer and MMA warps run their loops warp-wide and issue through elect.sync: issuing the
// asynchronous tensor ops from a converged warp is several times cheaper per op than from a single
// diverged lane.
// Scales arrive in the GEMM layout (512-byte atoms of 128 rows x 4 scale columns).  Every CTA loads
// the atoms of its own 128 A rows and of all 256 B rows, because each CTA's tensor core reads the A
// scales of its rows and the B scales of every column from its own TMEM.  The scale tensors are
// read through TMA maps, so atoms past the end of a tensor (the upper half of a pair tile past M)
// arrive as zeros.  For the grouped GEMM the A scales are in the grouped layout, where every expert
// group starts on a 128-row band, so a tile at an arbitrary row offset still reads whole atoms.
// Every mbarrier wait is bounded: on expiry the CTA records MX_ERR_TIMEOUT in a device word, stops
// issuing work and lets its in-flight copies land before the pair leaves and frees its TMEM.
#include "../../include/mxnum.h"
#include "mx_internal.h"
#include "mx_async.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

namespace mxk {

__device__ unsigned int g_mx_device_status = 0;

namespace {

constexpr int BM = 128;                   // rows per CTA (256 per pair)
constexpr int BKB = 128;                  // K bytes per pipeline stage
constexpr int NUM_THREADS = 320;         // producer, MMA, 8 epilogue warps
constexpr int TMEM_COLS = 512;
constexpr int MAX_GROUPS = MX_MAX_GROUPS;

struct Params {
    const uint8_t* sa; const uint8_t* sb;
    const float* alpha_a; int alpha_a_scope;
    const float* alpha_b; int alpha_b_scope;
    int64_t M, N, K;
    uint16_t* d; int64_t ldd;
    int64_t G; const int64_t* group_offsets;
    int64_t m_tiles, n_tiles, k_stages;
    int64_t nct;            // 4-column scale tiles per row band (same for A and B: same K)
    int64_t sb_group_bytes; // grouped: scale bytes per expert matrix
    int64_t total_tiles;    // dense
};

// ---------------------------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------------------------
using namespace async;

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int32_t c0, int32_t c1, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(map), "r"(c0), "r"(c1), "r"(src) : "memory");
}
// Load signalling an mbarrier that may sit in the peer CTA of the pair (cta_group::2 form).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1, uint32_t bar_cluster) {
    asm volatile("cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar_cluster) : "memory");
}
__device__ __forceinline__ uint32_t map_to_cta(uint32_t saddr, uint32_t cta_rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(cta_rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(bar_cluster) : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Bulk copy from this CTA's shared memory into another CTA's of the cluster, completing `bytes` on
// the destination CTA's mbarrier.
__device__ __forceinline__ void bulk_signal_copy(uint32_t dst_cluster, uint32_t src, uint32_t bytes, uint32_t bar_cluster) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst_cluster), "r"(src), "r"(bytes), "r"(bar_cluster) : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_group_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_group_read_n() { asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory"); }
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }


// Pair (cta_group::2) forms: issued by the even CTA of the pair, act on both CTAs' shared memory and
// TMEM at the same addresses; commits arrive on the barrier at the same offset in every CTA of `mask`.
__device__ __forceinline__ void tc2_commit_mc(uint32_t bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 :: "r"(bar), "h"(mask) : "memory");
}
__device__ __forceinline__ void tc2_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}
template <int FMT>
__device__ __forceinline__ void tc2_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t acc) {
    if (FMT == 0) {
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                     "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
                     :: "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc) : "memory");
    } else {
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                     "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
                     :: "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc) : "memory");
    }
}


// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128 bytes, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1 (bits 46..48), swizzle mode 2.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Descriptor of one 512-byte scale atom (32 rows x 16 bytes, contiguous, no swizzle).
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) |
           ((uint64_t)1 << 46);
}

// Instruction descriptor for the block-scaled kinds: B scale id (bits 4-5), A/B formats (7-9,
// 10-12), K-major A and B, N >> 3 (17-22), scale type (23: 1 = UE8M0, 0 = UE4M3), M >> 4 (24-28),
// A scale id (29-30).
template <int FMT, int MMA_M, int MMA_N>
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id) {
    const uint32_t fmt = FMT == 0 ? 0u : 1u;          // E4M3 (mxf8f6f4) / E2M1 (mxf4nvf4)
    const uint32_t scale_type = FMT == 0 ? 1u : 0u;
    return (sf_id << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(MMA_N >> 3) << 17) | (scale_type << 23) |
           ((uint32_t)(MMA_M >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float v[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------------------------
// Tile schedule (identical in every role)
// ---------------------------------------------------------------------------------------------
// Epilogue geometry: 8 warps, two per TMEM lane quadrant; warp (q, h) owns rows [32 q, 32 q + 32) of
// the CTA's 128 and columns [TN/2 h, TN/2 (h + 1)) of the tile.  Stores go out in 32-row x 16-column
// chunks (32-byte rows, 32-byte swizzle) through two 1 KB staging buffers per warp, or for short-K
// NVFP4 GEMMs in 32 x 64 chunks (128-byte rows, 128-byte swizzle) through one 4 KB buffer per warp.
constexpr int EPI_WARPS = 8;
constexpr int EPI_COLS = 16;
constexpr int EPI_BUF_BYTES = 32 * 2 * EPI_COLS;

// Second-level scales of this thread's row (loaded before the accumulator is ready).
template <bool GROUPED>
__device__ __forceinline__ void epilogue_alphas(const Params& p, int64_t row, bool row_ok, int64_t g, float& aa,
                                                float& ab_g) {
    aa = 1.0f;
    if (p.alpha_a_scope == 1) aa = __ldg(p.alpha_a);
    else if (p.alpha_a_scope == 2 && row_ok) aa = __ldg(p.alpha_a + row);
    ab_g = 1.0f;
    if (GROUPED && p.alpha_b_scope != 0) ab_g = __ldg(p.alpha_b + g);
    else if (!GROUPED && p.alpha_b_scope == 1) ab_g = __ldg(p.alpha_b);
}

// Drain of one tile by an epilogue warp: its 32 TMEM lanes x TN/2 FP32 columns (accumulator at tacc)
// into packed BF16 registers with the second-level scales applied; then TMEM is handed back by an
// arrival on a barrier of this CTA (`expect_signal`: the arrival also expects the odd CTA's 16-byte
// signal copy on the even CTA's barrier).
template <int TN, bool COL_ALPHA>
__device__ __forceinline__ void epilogue_drain(const Params& p, uint32_t tacc, int q, int h, int lane, int64_t n0,
                                               float aa, float ab_g, uint32_t tempty_bar, bool expect_signal,
                                               uint32_t (&packed)[TN / 4]) {
    constexpr int EPI_HALF = TN / 2;                // columns per epilogue warp
    const int64_t nh = n0 + h * EPI_HALF;           // first column of this warp's half
#pragma unroll
    for (int c = 0; c < EPI_HALF / 32; ++c) {
        float v[32];
        tmem_ld32(tacc + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * EPI_HALF + c * 32), v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float f0 = __fmul_rn(v[2 * i], aa), f1 = __fmul_rn(v[2 * i + 1], aa);
            if (COL_ALPHA) {
                const int64_t n = nh + c * 32 + 2 * i;
                f0 = __fmul_rn(f0, n < p.N ? __ldg(p.alpha_b + n) : 0.0f);
                f1 = __fmul_rn(f1, n + 1 < p.N ? __ldg(p.alpha_b + n + 1) : 0.0f);
            } else {
                f0 = __fmul_rn(f0, ab_g);
                f1 = __fmul_rn(f1, ab_g);
            }
            packed[c * 16 + i] = pack_bf16x2(f0, f1);
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
        if (expect_signal) mbar_arrive_expect_tx(tempty_bar, 16);
        else mbar_arrive(tempty_bar);
    }
}

// Stores of one drained tile slice: rows [row0 + 32 q, +32) that belong to the tile, columns of the
// warp's half.  TMA stores from the warp's two staging buffers at ebase, or plain 16-byte stores for
// a slice that straddles the end of an expert group.
template <int TN, bool GROUPED, int NBUF, int ECOLS>
__device__ __forceinline__ void epilogue_store(const Params& p, const CUtensorMap* tmD, int q, int h, int lane,
                                               int64_t row0, int64_t row_end, int64_t n0, uint32_t ebase,
                                               uint32_t& epi_chunk, const uint32_t (&packed)[TN / 4]) {
    constexpr int EPI_HALF = TN / 2;
    const int64_t row = row0 + q * 32 + lane;
    const bool row_ok = row < row_end;
    const int64_t nh = n0 + h * EPI_HALF;
    const int64_t wrow0 = row0 + q * 32;              // first row of this warp's slice
    if (wrow0 >= row_end) return;
    if (!GROUPED || wrow0 + 32 <= row_end) {
        // TMA stores; the tensor map clips rows >= M and columns >= N
        constexpr uint32_t BUF_BYTES = 32u * 2u * ECOLS;
        const uint32_t rbase_off = (uint32_t)(lane * 2 * ECOLS);
#pragma unroll
        for (int c = 0; c < EPI_HALF / ECOLS; ++c) {
            const int64_t col0 = nh + c * ECOLS;
            if (col0 < p.N) {
                const uint32_t buf = ebase + (epi_chunk % (uint32_t)NBUF) * BUF_BYTES;
                ++epi_chunk;
                // the store issued from this buffer NBUF chunks ago must have read it
                if (lane == 0) bulk_wait_group_read_n<NBUF - 1>();
                __syncwarp();
#pragma unroll
                for (int j = 0; j < ECOLS / 8; ++j) {
                    // 16-byte piece j of this row at its position under the 32- or 64-byte swizzle
                    // (the piece index XORed with address bit 7, or bits 7-8)
                    const uint32_t phys = ECOLS == 16 ? (uint32_t)j ^ ((uint32_t)(lane >> 2) & 1u)
                                        : ECOLS == 32 ? (uint32_t)j ^ ((uint32_t)(lane >> 1) & 3u)
                                                      : (uint32_t)j ^ ((uint32_t)lane & 7u);
                    const int pk = c * (ECOLS / 2) + 4 * j;
                    st_shared_v4(buf + rbase_off + 16u * phys, packed[pk], packed[pk + 1], packed[pk + 2], packed[pk + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(tmD, (int32_t)col0, (int32_t)wrow0, buf);
                    bulk_commit_group();
                }
            }
        }
    } else if (row_ok) {
        // the slice straddles the end of the expert group: the next group's rows belong to another
        // tile, so store this group's rows only (16-byte stores, N and ldd % 8 == 0)
        uint16_t* drow = p.d + row * p.ldd;
#pragma unroll
        for (int g8 = 0; g8 < EPI_HALF / 8; ++g8) {
            if (nh + g8 * 8 < p.N)
                *reinterpret_cast<uint4*>(drow + nh + g8 * 8) =
                    make_uint4(packed[4 * g8], packed[4 * g8 + 1], packed[4 * g8 + 2], packed[4 * g8 + 3]);
        }
    }
}

// ---------------------------------------------------------------------------------------------
// CTA-pair kernel: 256 x TN output tiles, each computed by the two CTAs of a cluster with the
// cta_group::2 MMA (M = 256, 128 rows in each CTA's TMEM; B split by N halves between the two CTAs'
// shared memory).  Each SM loads half of the B tile, so a stage carries less than a single-CTA tile
// for the same MMA work, and the ring holds more stages.
//   TN = 256: one accumulator (256 TMEM columns); long-K dense GEMMs, where the tile-boundary
//             drain is a small share of a tile
//   TN = 128: two accumulators (2 x 128 columns): the epilogue of tile i overlaps the MMAs of tile
//             i + 1; short-K grouped GEMMs, where a tile is only a few stages long
//   TN = 384: one accumulator of 384 columns filled by two MMAs per K step (N = 256 into columns
//             [0, 256), N = 128 into [256, 384)); dense MXFP8 only (the NVFP4 scale columns of a
//             stage would not fit next to it in TMEM).  Each CTA holds B rows [128 r, +128) and
//             [256 + 64 r, +64) of the tile, so both MMAs find their B halves and their B scale
//             bands (128-row atoms 0-1 and 2) whole
//   both CTAs  warp 0: TMA loads of this CTA's A rows, B half and scale atoms (the B scales of all
//              TN columns, which each CTA's tensor core reads from its own TMEM); every load
//              signals the stage barrier in the even (leader) CTA
//   leader     warp 1: tcgen05.cp (each CTA's atoms into its own TMEM) and tcgen05.mma for the pair;
//              commits arrive on the barriers of both CTAs
//   both CTAs  warps 2..9: epilogue of this CTA's 128 rows; TMEM release arrives in the leader
// ---------------------------------------------------------------------------------------------
template <int FMT, bool GROUPED, int TN, int EV = 0>
struct PairCfg {
    static_assert(TN == 128 || TN == 256 || TN == 384, "tile width");
    static_assert(TN != 384 || (FMT == 0 && !GROUPED), "384-column tiles: dense MXFP8 only");
    static constexpr int ACC = TN == 128 ? 2 : 1;          // accumulator buffers
    // ring depth within the shared-memory budget (the grouped tables take 16.5 KB)
    static constexpr int NST = TN == 384 ? 5
                             : FMT == 0 ? (TN == 256 ? (GROUPED ? 5 : 6) : (GROUPED ? 6 : 8))
                                        : (TN == 256 ? 5 : (GROUPED ? 6 : 7));
    // rows per B load: 384-column tiles load each CTA's 192 rows as three 64-row boxes (128 rows for
    // the N = 256 MMA, 64 for the N = 128 MMA), the other widths one box of TN / 2 rows
    static constexpr int B_BOX = TN == 384 ? 64 : TN / 2;
    // epilogue staging buffers per warp (one for 384-column tiles, so that a fifth stage fits)
    // epilogue stores: EV = 0, 32-row x 16-column chunks through two 1 KB buffers per warp; EV = 3,
    // 32 x 64 chunks (128-byte rows, 128-byte swizzle) through one 4 KB buffer per warp
    static constexpr int EPI_NBUF = TN == 384 ? 1 : (EV == 3 ? 1 : 2);
    static constexpr int EPI_C = EV == 3 ? 64 : EPI_COLS;   // columns per staged store
    static constexpr int EPI_BUF = 32 * 2 * EPI_C;
    static constexpr int SF_ATOMS_A = FMT == 0 ? 1 : 4;
    static constexpr int SFB_BANDS = TN / 128;
    static constexpr int SFA_BYTES = 512 * SF_ATOMS_A;     // this CTA's 128 rows
    static constexpr int SFB_BYTES = SFB_BANDS * SFA_BYTES; // all TN columns
    static constexpr int SFA_COLS = 4 * SF_ATOMS_A;
    static constexpr int SFB_COLS = SFB_BANDS * SFA_COLS;
    static constexpr int TMEM_SF = ACC * TN;                // scale slots after the accumulators
    static constexpr int A_BYTES = 128 * BKB;
    static constexpr int B_BYTES = (TN / 2) * BKB;
    static constexpr uint32_t STAGE_TX = 2u * (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES);   // both CTAs
    static constexpr int SMEM_A = 0;
    static constexpr int SMEM_B = SMEM_A + NST * A_BYTES;
    static constexpr int SMEM_SFA = SMEM_B + NST * B_BYTES;
    static constexpr int SMEM_SFB = SMEM_SFA + NST * SFA_BYTES;
    static constexpr int SMEM_EPI = (SMEM_SFB + NST * SFB_BYTES + 1023) / 1024 * 1024;
    static constexpr int SMEM_BAR = SMEM_EPI + EPI_WARPS * EPI_NBUF * EPI_BUF;
    static constexpr int SMEM_MISC = SMEM_BAR + 8 * (2 * NST + 7);
    static constexpr int SMEM_SIGNAL = (SMEM_MISC + 16 + 15) / 16 * 16;   // 16-byte signal source / target
    static constexpr int SMEM_TABLES = SMEM_SIGNAL + 16;   // grouped: row offsets, pair-tile and band prefixes
    // grouped: the tables hold G + 1 entries each, so the launch sizes them by G (table_bytes)
    static constexpr int table_bytes(int64_t G) { return GROUPED ? (int)(8 * (G + 1) + 4 * (2 * (G + 1) + 32)) : 0; }
    static constexpr int smem_alloc(int64_t G) { return SMEM_TABLES + table_bytes(G) + 1024; }
    static constexpr int SMEM_LIMIT = 227 * 1024;
    // the most groups whose tables fit (all of MX_MAX_GROUPS with the narrow staging)
    static constexpr int64_t MAX_G = GROUPED ? (SMEM_LIMIT - 1024 - SMEM_TABLES - 4 * 32 - 8 - 8) / 16 : 0;
    static constexpr int SMEM_ALLOC = smem_alloc(GROUPED ? 1 : 0);
    static_assert(SMEM_B % 1024 == 0 && SMEM_EPI % 1024 == 0, "operand and staging alignment");
    static_assert(TMEM_SF + NST * (SFA_COLS + SFB_COLS) <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

struct PairTile {
    int64_t row0, row_end;   // this CTA's rows [row0, row0 + 128), real below row_end
    int64_t n0;              // first output column of the pair tile
    int64_t g;               // group (grouped GEMM) or 0
    int64_t band_a;          // 128-row band of A's scale layout holding this CTA's rows
};

// Dense: bands of 8 pair rows (16 M-tiles); inside a band N-tiles advance every 8 pair tiles.
template <int TN>
__device__ __forceinline__ PairTile pair_dense_tile(const Params& p, int64_t t, uint32_t rank) {
    constexpr int64_t GM = 8;
    const int64_t band_tiles = GM * p.n_tiles;
    const int64_t band = t / band_tiles, in = t % band_tiles;
    const int64_t band_m = min64(GM, p.m_tiles - band * GM);
    const int64_t mp = band * GM + in % band_m, nt = in / band_m;
    PairTile r;
    r.row0 = mp * 256 + 128 * (int64_t)rank; r.row_end = p.M; r.n0 = nt * TN; r.g = 0;
    r.band_a = mp * 2 + rank;
    return r;
}

// Grouped: s_off = the group row offsets, ptile2[g] = pair tiles (256 rows) of groups < g, pband[g] =
// 128-row bands of groups < g (group g's first band in the grouped scale layout); all in shared memory.
template <int TN>
__device__ __forceinline__ PairTile pair_grouped_tile(const Params& p, const int64_t* s_off, const int* ptile2,
                                                      const int* pband, int64_t t, uint32_t rank) {
    const int64_t mt_global = t / p.n_tiles;
    int lo = 0, hi = (int)p.G;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ptile2[mid] <= mt_global) lo = mid; else hi = mid;
    }
    const int64_t g = lo;
    const int64_t pm = mt_global - ptile2[g];
    PairTile r;
    r.row0 = s_off[g] + pm * 256 + 128 * (int64_t)rank;
    r.row_end = s_off[g + 1];
    r.n0 = (t % p.n_tiles) * TN;
    r.g = g;
    r.band_a = pband[g] + 2 * pm + rank;
    return r;
}

template <int FMT, bool GROUPED, bool COL_ALPHA, int TN, int EV>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
bs_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                    const __grid_constant__ CUtensorMap tmD, const Params p) {
    using C = PairCfg<FMT, GROUPED, TN, EV>;
    constexpr int NST = C::NST;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + C::SMEM_BAR;                 // NST barriers (used in the leader)
    const uint32_t bar_empty = bar_full + 8 * NST;                 // NST barriers
    const uint32_t bar_tfull = bar_empty + 8 * NST;                // 2 barriers (one per accumulator)
    const uint32_t bar_tempty = bar_tfull + 16;                    // 2 barriers (used in the leader)
    const uint32_t bar_done = bar_tempty + 16;
    const uint32_t bar_tempty_odd = bar_done + 8;                  // 2 barriers (odd CTA): its epilogue drained
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SMEM_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::SMEM_MISC + 4);
    int64_t* s_off = reinterpret_cast<int64_t*>(smem + C::SMEM_TABLES);
    int* ptile2 = reinterpret_cast<int*>(s_off + (p.G + 1));
    int* pband = ptile2 + (p.G + 1);
    int* s_warp = pband + (p.G + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tfull + 8 * b, 1);
            // the even CTA's epilogue warps (one of them also expects the odd CTA's 16-byte signal)
            mbar_init(bar_tempty + 8 * b, EPI_WARPS);
            mbar_init(bar_tempty_odd + 8 * b, EPI_WARPS);
        }
        mbar_init(bar_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmA) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmB) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmSA) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmSB) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmD) : "memory");
    }
    if (warp == 1) {
        // one allocation for the pair, made by a warp of each CTA together
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    if (GROUPED) {
        for (int i = threadIdx.x; i <= (int)p.G; i += blockDim.x) s_off[i] = __ldg(p.group_offsets + i);
        __syncthreads();
        scan_group_tiles<256>(s_off, (int)p.G, ptile2, s_warp);
        scan_group_tiles<128>(s_off, (int)p.G, pband, s_warp);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                       // barriers of both CTAs initialised before any signal
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int64_t total_tiles = GROUPED ? (int64_t)ptile2[p.G] * p.n_tiles : p.total_tiles;
    const int64_t pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

    if (warp == 0) {
        // ------------------------------- producer (both CTAs) -------------------------------
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs) {
            const PairTile tile = GROUPED ? pair_grouped_tile<TN>(p, s_off, ptile2, pband, t, rank) : pair_dense_tile<TN>(p, t, rank);
            const int64_t brow = (GROUPED ? tile.g * p.N : 0) + tile.n0 + (TN / 2) * (int64_t)rank;
            const int64_t sfb_y0 = GROUPED ? tile.g * (p.sb_group_bytes >> 8) : 0;   // 256-byte rows
            const int64_t bt0 = tile.n0 / 128;
            for (int64_t ks = 0; ks < p.k_stages; ++ks) {
                if (!warp_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag, &g_mx_device_status)) { ok = false; break; }
                if (elect_one()) {
                    const uint32_t fb = map_to_cta(bar_full + 8 * stage, 0);
                    if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, C::STAGE_TX);
                    const uint32_t sA = sbase + C::SMEM_A + stage * C::A_BYTES;
                    const uint32_t sB = sbase + C::SMEM_B + stage * C::B_BYTES;
                    const uint32_t sSFA = sbase + C::SMEM_SFA + stage * C::SFA_BYTES;
                    const uint32_t sSFB = sbase + C::SMEM_SFB + stage * C::SFB_BYTES;
                    const int64_t ct0 = ks * C::SF_ATOMS_A;
                    const int32_t kb = (int32_t)(ks * BKB);
                    tma_load_2d_pair(sA, &tmA, kb, (int32_t)tile.row0, fb);
                    if (TN == 384) {
                        // the N = 256 MMA takes columns [128 rank, +128) of the tile from this CTA,
                        // the N = 128 MMA columns [256 + 64 rank, +64)
                        const int64_t b0 = tile.n0 + 128 * (int64_t)rank;
                        tma_load_2d_pair(sB, &tmB, kb, (int32_t)b0, fb);
                        tma_load_2d_pair(sB + 64 * BKB, &tmB, kb, (int32_t)(b0 + 64), fb);
                        tma_load_2d_pair(sB + 128 * BKB, &tmB, kb, (int32_t)(tile.n0 + 256 + 64 * (int64_t)rank), fb);
                    } else {
                        tma_load_2d_pair(sB, &tmB, kb, (int32_t)brow, fb);
                    }
                    // scale atoms: 512 bytes = two 256-byte rows of the scale maps; bands past the
                    // end of a tensor read as zeros
                    tma_load_2d_pair(sSFA, &tmSA, 0, (int32_t)((tile.band_a * p.nct + ct0) * 2), fb);
#pragma unroll
                    for (int hb = 0; hb < C::SFB_BANDS; ++hb)
                        tma_load_2d_pair(sSFB + hb * C::SFA_BYTES, &tmSB, 0,
                                         (int32_t)(sfb_y0 + ((bt0 + hb) * p.nct + ct0) * 2), fb);
                }
                __syncwarp();
                if (++stage == NST) { stage = 0; phase ^= 1; }
            }
        }
        if (!ok && lane == 0) *abort_flag = 1;
    } else if (warp == 1) {
        // ------------------------------- scale copies + MMA (leader) -------------------------------
        if (leader) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, issued_any = false;
            int64_t ti = 0;                           // this pair's tile count: accumulator ti % ACC
            for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs, ++ti) {
                const uint32_t ab = (uint32_t)(ti % C::ACC);
                const uint32_t use = (uint32_t)(ti / C::ACC);        // uses of this accumulator so far
                if (!warp_wait(bar_tempty + 8 * ab, (use & 1u) ^ 1u, abort_flag, &g_mx_device_status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t tacc = tmem + ab * TN;
                for (int64_t ks = 0; ks < p.k_stages; ++ks) {
                    if (!warp_wait(bar_full + 8 * stage, phase, abort_flag, &g_mx_device_status)) { ok = false; break; }
                    tc_fence_after();
                    if (elect_one()) {
                        const uint32_t sA = sbase + C::SMEM_A + stage * C::A_BYTES;
                        const uint32_t sB = sbase + C::SMEM_B + stage * C::B_BYTES;
                        const uint32_t sSFA = sbase + C::SMEM_SFA + stage * C::SFA_BYTES;
                        const uint32_t sSFB = sbase + C::SMEM_SFB + stage * C::SFB_BYTES;
                        const uint32_t tSFA = tmem + C::TMEM_SF + stage * (C::SFA_COLS + C::SFB_COLS);
                        const uint32_t tSFB = tSFA + C::SFA_COLS;
                        // A atom j to columns 4j..4j+3; B band h, atom j to SFB_BANDS * 4j + 4h
#pragma unroll
                        for (int j = 0; j < C::SF_ATOMS_A; ++j) {
                            tc2_cp_sf(tSFA + 4 * j, desc_sf(sSFA + 512 * j));
#pragma unroll
                            for (int hb = 0; hb < C::SFB_BANDS; ++hb)
                                tc2_cp_sf(tSFB + C::SFB_BANDS * 4 * j + 4 * hb, desc_sf(sSFB + hb * C::SFA_BYTES + 512 * j));
                        }
#pragma unroll
                        for (int j = 0; j < BKB / 32; ++j) {
                            // MXFP8: one atom covers the 4 MMAs of the stage, the scale id picks the byte;
                            // NVFP4: each MMA (K = 64) consumes a whole atom word
                            const uint32_t sf_id = FMT == 0 ? (uint32_t)j : 0u;
                            const uint32_t col = FMT == 0 ? 0u : (uint32_t)j;
                            const uint32_t accum = (ks > 0 || j > 0) ? 1u : 0u;
                            if (TN == 384) {
                                // columns [0, 256) from the first 128 B rows of each CTA (scale bands 0
                                // and 1), columns [256, 384) from the next 64 (band 2)
                                tc2_mma<FMT>(tacc, desc_sw128(sA + 32 * j), desc_sw128(sB + 32 * j),
                                             make_idesc<FMT, 2 * BM, 256>(sf_id), tSFA + 4 * col,
                                             tSFB + C::SFB_BANDS * 4 * col, accum);
                                tc2_mma<FMT>(tacc + 256, desc_sw128(sA + 32 * j), desc_sw128(sB + 128 * BKB + 32 * j),
                                             make_idesc<FMT, 2 * BM, 128>(sf_id), tSFA + 4 * col,
                                             tSFB + C::SFB_BANDS * 4 * col + 8, accum);
                            } else {
                                tc2_mma<FMT>(tacc, desc_sw128(sA + 32 * j), desc_sw128(sB + 32 * j),
                                             make_idesc<FMT, 2 * BM, TN>(sf_id), tSFA + 4 * col,
                                             tSFB + C::SFB_BANDS * 4 * col, accum);
                            }
                        }
                        tc2_commit_mc(bar_empty + 8 * stage, (uint16_t)3);
                    }
                    __syncwarp();
                    issued_any = true;
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                if (elect_one()) tc2_commit_mc(bar_tfull + 8 * ab, (uint16_t)3);
                __syncwarp();
            }
            // the odd CTA's last TMEM-release copies land on these barriers after the final MMAs: wait for
            // them, so that neither CTA leaves while a copy into or out of its shared memory is in flight
            for (int b = 0; b < C::ACC && ok; ++b) {
                const int64_t uses = (ti - b + C::ACC - 1) / C::ACC;
                if (uses > 0 && !warp_wait(bar_tempty + 8 * b, (uint32_t)((uses - 1) & 1), abort_flag, &g_mx_device_status))
                    ok = false;
            }
            if (issued_any) {
                // the pair's MMAs read the peer's shared memory: all of them complete before either
                // CTA leaves the final cluster barrier
                if (elect_one()) {
                    tc2_commit_mc(bar_done, (uint16_t)1);
                    const unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(bar_done, 0) && globaltimer() - t0 < WAIT_LIMIT_NS) {}
                }
                __syncwarp();
            }
        } else {
            // odd CTA: each time its epilogue warps have drained a tile (a local barrier), a 16-byte bulk
            // copy completes on the even CTA's TMEM-empty barrier (cluster-scope release arrivals from
            // each epilogue warp stall their warps for thousands of cycles)
            const uint32_t tempty_leader = map_to_cta(bar_tempty, 0);
            const uint32_t sig_dst = map_to_cta(sbase + C::SMEM_SIGNAL, 0);
            bool ok = true;
            int64_t ti = 0;
            for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs, ++ti) {
                const uint32_t ab = (uint32_t)(ti % C::ACC);
                const uint32_t use = (uint32_t)(ti / C::ACC);
                if (!warp_wait(bar_tempty_odd + 8 * ab, use & 1u, abort_flag, &g_mx_device_status)) { ok = false; break; }
                if (lane == 0) bulk_signal_copy(sig_dst, sbase + C::SMEM_SIGNAL, 16, tempty_leader + 8 * ab);
                __syncwarp();
            }
            if (!ok && lane == 0) *abort_flag = 1;
        }
    } else {
        // ------------------------------- epilogue (both CTAs) -------------------------------
        const int q = warp & 3;                     // TMEM lane quadrant this warp may access
        const int h = (warp - 2) >> 2;              // column half
        const uint32_t tempty_mine = leader ? bar_tempty : bar_tempty_odd;
        const uint32_t ebase = sbase + C::SMEM_EPI + (uint32_t)((warp - 2) * C::EPI_NBUF * C::EPI_BUF);
        uint32_t epi_chunk = 0;
        // tile coordinates and row scales of the next tile are fetched while this tile's stores run
        PairTile tile{};
        float aa = 1.0f, ab_g = 1.0f;
        if (pair_id < total_tiles) {
            tile = GROUPED ? pair_grouped_tile<TN>(p, s_off, ptile2, pband, pair_id, rank) : pair_dense_tile<TN>(p, pair_id, rank);
            const int64_t row = tile.row0 + q * 32 + lane;
            epilogue_alphas<GROUPED>(p, row, row < tile.row_end, tile.g, aa, ab_g);
        }
        int64_t ti = 0;
        for (int64_t t = pair_id; t < total_tiles; t += n_pairs, ++ti) {
            const uint32_t ab = (uint32_t)(ti % C::ACC);
            const uint32_t use = (uint32_t)(ti / C::ACC);
            if (!mbar_wait(bar_tfull + 8 * ab, use & 1u, abort_flag, &g_mx_device_status)) break;
            tc_fence_after();
            uint32_t packed[TN / 4];
            epilogue_drain<TN, COL_ALPHA>(p, tmem + ab * TN, q, h, lane, tile.n0, aa, ab_g, tempty_mine + 8 * ab,
                                          leader && warp == 2, packed);
            const PairTile cur = tile;
            const int64_t tn = t + n_pairs;
            if (tn < total_tiles) {
                tile = GROUPED ? pair_grouped_tile<TN>(p, s_off, ptile2, pband, tn, rank) : pair_dense_tile<TN>(p, tn, rank);
                const int64_t row = tile.row0 + q * 32 + lane;
                epilogue_alphas<GROUPED>(p, row, row < tile.row_end, tile.g, aa, ab_g);
            }
            epilogue_store<TN, GROUPED, C::EPI_NBUF, C::EPI_C>(p, &tmD, q, h, lane, cur.row0, cur.row_end, cur.n0, ebase, epi_chunk, packed);
        }
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // after an expired wait: give loads already issued by this CTA time to land before exit
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {}
    }
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
}

// ---------------------------------------------------------------------------------------------
// Dequantize-in-mainloop BF16 GEMM (the dequantized backward of the 4-bitter page: the backward
// GEMMs take BF16 operands rebuilt from the forward's NVFP4 values, y = x * DQ(Q(w))):
//   D[m, n] = BF16( alpha_a[m] * sum_k A[m, k] * DQ(B)[n, k] ),
//   DQ(B)[n, k] = BF16( fp32(val(q) * val(bs)) * S ),  S per B tensor or per B row,
// i.e. exactly the values mx_dequantize_bf16 would write, without that BF16 copy of B in HBM: B is
// read as NVFP4 codes + E4M3 scales and expanded in shared memory.  Same CTA-pair structure as the
// block-scaled kernel (256 x 256 tiles, tcgen05.mma.cta_group::2, here kind::f16 with BF16 operands
// and FP32 accumulation), two accumulators (512 TMEM columns) so the drain of one tile overlaps the
// next tile's MMAs, and four converter warps per CTA:
//   warp 0        TMA: A (BF16, 128 rows x 64 values per stage) signalling the even CTA's stage
//                 barrier; this CTA's 128 B rows of codes (32 bytes each) and their scale atom into
//                 a local barrier
//   warp 1        (even CTA) the pair MMAs, 4 per stage (K = 16 each)
//   warps 2..9    epilogue (32-column chunks: tcgen05.ld, row factor, BF16, TMA store)
//   warps 10..13  converters: thread r expands B row r of this CTA's half for the stage (64 values:
//                 E2M1 pairs to FP16, exact product with the FP16 block scale, times S in FP32,
//                 round to BF16) into the 128-byte-swizzled K-major tile the MMA descriptor expects,
//                 fences the generic-proxy writes for the tensor core and arrives (one lane per warp)
//                 on a barrier of its own CTA: the even CTA's stage barrier directly; in the odd CTA a
//                 local barrier that warp 1 (idle there) forwards to the even CTA's stage barrier as the
//                 completion of a 16-byte bulk copy
// ---------------------------------------------------------------------------------------------
constexpr int DQ_CONV_WARPS = 8;                           // converter warps per CTA (2 per scheduler)
constexpr int DQ_CONV_WARP0 = 10;
constexpr int DQ_QPROD_WARP = DQ_CONV_WARP0 + DQ_CONV_WARPS;   // the codes producer
constexpr int DQ_THREADS = 32 * (DQ_QPROD_WARP + 1);
constexpr int DQ_TN = 256;
constexpr int DQ_CONV_CHUNKS = 8 * 4 / DQ_CONV_WARPS;          // 16-byte BF16 chunks per converter thread
static_assert(DQ_CONV_CHUNKS == 2 || DQ_CONV_CHUNKS == 4 || DQ_CONV_CHUNKS == 8, "converter split");

struct DqParams {
    const float* alpha_a; int alpha_a_scope;
    const float* sb2; int sb2_scope;        // B's FP32 second-level scale: 1 = one value, 2 = per B row,
                                            // 3 = per K index (per-token scales of a weight-gradient B)
    int64_t M, N, K;
    uint16_t* d; int64_t ldd;
    int64_t m_tiles, n_tiles, k_stages, nct, total_tiles;
};

template <bool WG>
struct DqCfg {
    static constexpr int NST = 4;                          // A / B (BF16) ring
    static constexpr int NQ = 3;                           // codes ring
    static constexpr int A_BLOCK = 128 * BKB;              // 128 rows x 64 BF16
    static constexpr int A_BYTES = 2 * A_BLOCK;            // this CTA's rows of both 256-row halves of the tile
    static constexpr int B_BYTES = 128 * BKB;              // this CTA's 128 B rows x 64 BF16 (built here)
    static constexpr int Q_BYTES = 128 * 32;               // their codes, 64 E2M1 values per row
    // their scales: one atom (4 scales per row) for K-major B; for the weight gradient (B = X, tokens
    // along K) the two atoms holding the 8 block columns of the CTA's 128 B rows for 128 tokens
    static constexpr int SF_BYTES = WG ? 1024 : 512;
    static constexpr uint32_t A_TX = 2u * A_BYTES;         // both CTAs' A rows, on the even CTA's barrier
    static constexpr uint32_t Q_TX = Q_BYTES + SF_BYTES;   // per CTA, on its own barrier
    static constexpr int FULL_ARRIVALS = 1 + DQ_CONV_WARPS;      // producer and the even CTA's converter warps
    static constexpr uint32_t SIGNAL_TX = 16;                    // the odd CTA's per-stage signal copy
    static constexpr int SMEM_A = 0;
    static constexpr int SMEM_B = SMEM_A + NST * A_BYTES;
    static constexpr int SMEM_Q = SMEM_B + NST * B_BYTES;
    static constexpr int SMEM_SF = SMEM_Q + NQ * Q_BYTES;
    static constexpr int SMEM_EPI = (SMEM_SF + NQ * SF_BYTES + 1023) / 1024 * 1024;
    static constexpr int SMEM_BAR = SMEM_EPI + EPI_WARPS * 2 * EPI_BUF_BYTES;
    static constexpr int SMEM_MISC = SMEM_BAR + 8 * (3 * NST + 2 * NQ + 5);
    static constexpr int SMEM_SIGNAL = (SMEM_MISC + 16 + 15) / 16 * 16;   // 16-byte target / source
    static constexpr int SMEM_ALLOC = SMEM_SIGNAL + 16 + 1024;
    static_assert(SMEM_B % 1024 == 0 && SMEM_Q % 1024 == 0 && SMEM_EPI % 1024 == 0, "alignment");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// Output tiles of 512 rows x 256 columns: the pair runs two M = 256 MMAs per K step on the same
// converted B tile (rows [m0, m0 + 256) and [m0 + 256, m0 + 512), CTA r holding rows 128 r + [0, 128)
// of each half), so each expanded B value feeds twice the tensor work.  Bands of 8 row tiles; inside
// a band N-tiles advance every 8 tiles.
__device__ __forceinline__ PairTile dq_tile(const DqParams& p, int64_t t, uint32_t rank) {
    constexpr int64_t GM = 8;
    const int64_t band_tiles = GM * p.n_tiles;
    const int64_t band = t / band_tiles, in = t % band_tiles;
    const int64_t band_m = min64(GM, p.m_tiles - band * GM);
    const int64_t mp = band * GM + in % band_m, nt = in / band_m;
    PairTile r;
    r.row0 = mp * 512 + 128 * (int64_t)rank; r.row_end = p.M; r.n0 = nt * DQ_TN; r.g = 0; r.band_a = 0;
    return r;
}

// kind::f16 instruction descriptor: D FP32 (bits 4-5 = 1), A and B BF16 (7-9, 10-12 = 1), K-major
// A and B, N >> 3 (17-22), M >> 4 (24-28).
template <int MMA_M, int MMA_N, bool MN_MAJOR = false>
__device__ __forceinline__ uint32_t make_idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((MN_MAJOR ? 1u : 0u) << 15) | ((MN_MAJOR ? 1u : 0u) << 16) |
           ((uint32_t)(MMA_N >> 3) << 17) | ((uint32_t)(MMA_M >> 4) << 24);
}

// Shared-memory matrix descriptor, MN-major, 128-byte swizzle (16-bit elements): atoms of 64 MN
// elements (one 128-byte row) x 8 K rows; MN atoms DQ_MN_ATOM bytes apart (leading byte offset), 8-row
// K groups 1024 bytes apart (stride byte offset).
constexpr int DQ_MN_ATOM = 64 * 128;
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(DQ_MN_ATOM >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tc2_mma_bf16(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
}

// One E4M3 scale byte -> the same FP16 value in both halves (exact).
__device__ __forceinline__ uint32_t e4m3_to_f16x2_bcast(uint32_t byte) {
    uint32_t r;
    asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(r) : "r"(byte * 0x0101u));
    return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Eight E2M1 codes (one word, element 0 in the low nibble) of one 16-block -> four BF16 pairs:
// BF16(fp32(val(q) * val(bs)) * S).  val(q) * val(bs) has at most 6 significant bits and lies in
// [2^-10, 2688], so the FP16 product is exact and equals the FP32 one.
__device__ __forceinline__ uint4 dq_word(uint32_t w, uint32_t bs_h2, float S) {
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t prod = hmul2_u32(e2m1x2_to_f16x2((w >> (8 * j)) & 0xFFu), bs_h2);
        const float f0 = __half2float(__ushort_as_half((unsigned short)(prod & 0xFFFFu)));
        const float f1 = __half2float(__ushort_as_half((unsigned short)(prod >> 16)));
        o[j] = pack_bf16x2(__fmul_rn(f0, S), __fmul_rn(f1, S));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}



template <bool WG>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(DQ_THREADS, 1)
dq_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmSB, const __grid_constant__ CUtensorMap tmD,
                    const DqParams p) {
    using C = DqCfg<WG>;
    constexpr int NST = C::NST;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + C::SMEM_BAR;            // NST (even CTA): A bytes + converters + signal
    const uint32_t bar_empty = bar_full + 8 * NST;            // NST (each CTA): the stage's MMAs are done
    const uint32_t bar_bconv = bar_empty + 8 * NST;           // NST (odd CTA): its converter warps are done
    const uint32_t bar_qfull = bar_bconv + 8 * NST;           // NQ (each CTA): codes + scale atom landed
    const uint32_t bar_qempty = bar_qfull + 8 * C::NQ;        // NQ (each CTA): the converters have read them
    const uint32_t bar_tfull = bar_qempty + 8 * C::NQ;        // 2
    const uint32_t bar_tempty = bar_tfull + 16;               // 2 (even CTA)
    const uint32_t bar_done = bar_tempty + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SMEM_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::SMEM_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar_full + 8 * s, C::FULL_ARRIVALS);
            mbar_init(bar_empty + 8 * s, 1);
            mbar_init(bar_bconv + 8 * s, DQ_CONV_WARPS);
        }
        for (int s = 0; s < C::NQ; ++s) {
            mbar_init(bar_qfull + 8 * s, 1);
            mbar_init(bar_qempty + 8 * s, DQ_CONV_WARPS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tfull + 8 * b, 1);
            mbar_init(bar_tempty + 8 * b, 2 * EPI_WARPS);
        }
        mbar_init(bar_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmA) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmQ) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmSB) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmD) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int64_t total_tiles = p.total_tiles;
    const int64_t pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

    if (warp == 0) {
        // ------------------------------- producer (both CTAs) -------------------------------
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs) {
            const PairTile tile = dq_tile(p, t, rank);
            for (int64_t ks = 0; ks < p.k_stages; ++ks) {
                if (!warp_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag, &g_mx_device_status)) { ok = false; break; }
                if (elect_one()) {
                    const uint32_t fb = map_to_cta(bar_full + 8 * stage, 0);
                    if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, C::A_TX + C::SIGNAL_TX);
                    const uint32_t sA = sbase + C::SMEM_A + stage * C::A_BYTES;
                    if constexpr (WG) {
                        // A = dY^T: boxes of 64 tokens x 64 output features of dY [T, O] (MN-major)
#pragma unroll
                        for (int b = 0; b < 2; ++b)
#pragma unroll
                            for (int j = 0; j < 2; ++j)
                                tma_load_2d_pair(sA + b * C::A_BLOCK + j * DQ_MN_ATOM, &tmA,
                                                 (int32_t)(tile.row0 + 256 * b + 64 * j), (int32_t)(ks * 64), fb);
                    } else {
                        tma_load_2d_pair(sA, &tmA, (int32_t)(ks * BKB), (int32_t)tile.row0, fb);
                        tma_load_2d_pair(sA + C::A_BLOCK, &tmA, (int32_t)(ks * BKB), (int32_t)(tile.row0 + 256), fb);
                    }
                }
                __syncwarp();
                if (++stage == NST) { stage = 0; phase ^= 1; }
            }
        }
        if (!ok && lane == 0) *abort_flag = 1;
    } else if (warp == 1) {
        // ------------------------------- MMA (even CTA) -------------------------------
        if (leader) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, issued_any = false;
            int64_t ti = 0;
            for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs, ++ti) {
                // both accumulators (rows m0 + [0, 256) and m0 + [256, 512)) fill all 512 TMEM columns
                if (!warp_wait(bar_tempty, ((uint32_t)ti & 1u) ^ 1u, abort_flag, &g_mx_device_status)) { ok = false; break; }
                tc_fence_after();
                for (int64_t ks = 0; ks < p.k_stages; ++ks) {
                    if (!warp_wait(bar_full + 8 * stage, phase, abort_flag, &g_mx_device_status)) { ok = false; break; }
                    tc_fence_after();
                    if (elect_one()) {
                        const uint32_t sA = sbase + C::SMEM_A + stage * C::A_BYTES;
                        const uint32_t sB = sbase + C::SMEM_B + stage * C::B_BYTES;
#pragma unroll
                        for (int j = 0; j < BKB / 32; ++j) {
                            // K = 16 per MMA: 32 bytes along a K-major row, or two 8-row K groups MN-major
                            const uint32_t koff = WG ? 2048u * j : 32u * j;
                            const uint64_t bd = WG ? desc_mn_sw128(sB + koff) : desc_sw128(sB + koff);
                            const uint64_t ad0 = WG ? desc_mn_sw128(sA + koff) : desc_sw128(sA + koff);
                            const uint64_t ad1 = WG ? desc_mn_sw128(sA + C::A_BLOCK + koff) : desc_sw128(sA + C::A_BLOCK + koff);
                            const uint32_t acc = (ks > 0 || j > 0) ? 1u : 0u;
                            tc2_mma_bf16(tmem, ad0, bd, make_idesc_bf16<2 * BM, DQ_TN, WG>(), acc);
                            tc2_mma_bf16(tmem + DQ_TN, ad1, bd, make_idesc_bf16<2 * BM, DQ_TN, WG>(), acc);
                        }
                        tc2_commit_mc(bar_empty + 8 * stage, (uint16_t)3);
                    }
                    __syncwarp();
                    issued_any = true;
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                if (elect_one()) tc2_commit_mc(bar_tfull, (uint16_t)3);
                __syncwarp();
            }
            if (issued_any) {
                if (elect_one()) {
                    tc2_commit_mc(bar_done, (uint16_t)1);
                    const unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(bar_done, 0) && globaltimer() - t0 < WAIT_LIMIT_NS) {}
                }
                __syncwarp();
            }
        } else {
            // odd CTA: once all of this CTA's converter warps have finished a stage (they arrive on a
            // local barrier), a 16-byte bulk copy into the even CTA completes SIGNAL_TX bytes on its
            // stage barrier.  The copy is an asynchronous-proxy operation ordered after the converters'
            // fenced writes, and issuing it does not block (a cluster-scope release arrival stalled the
            // issuing thread ~1-2k cycles per stage and starved the tensor core).
            const uint32_t full_leader = map_to_cta(bar_full, 0);
            const uint32_t sig_dst = map_to_cta(sbase + C::SMEM_SIGNAL, 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs) {
                for (int64_t ks = 0; ks < p.k_stages; ++ks) {
                    if (!warp_wait(bar_bconv + 8 * stage, phase, abort_flag, &g_mx_device_status)) { ok = false; break; }
                    if (lane == 0) bulk_signal_copy(sig_dst, sbase + C::SMEM_SIGNAL, C::SIGNAL_TX, full_leader + 8 * stage);
                    __syncwarp();
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && lane == 0) *abort_flag = 1;
        }
    } else if (warp < DQ_CONV_WARP0) {
        // ------------------------------- epilogue (both CTAs) -------------------------------
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const uint32_t tempty_leader = map_to_cta(bar_tempty, 0);
        const uint32_t ebase = sbase + C::SMEM_EPI + (uint32_t)((warp - 2) * 2 * EPI_BUF_BYTES);
        uint32_t epi_chunk = 0;
        int64_t ti = 0;
        for (int64_t t = pair_id; t < total_tiles; t += n_pairs, ++ti) {
            const PairTile tile = dq_tile(p, t, rank);
            if (!mbar_wait_backoff(bar_tfull, (uint32_t)ti & 1u, abort_flag, &g_mx_device_status)) break;
            tc_fence_after();
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                const int64_t wrow0 = tile.row0 + 256 * half + q * 32;
                const int64_t row = wrow0 + lane;
                float aa = 1.0f;
                if (p.alpha_a_scope == 1) aa = __ldg(p.alpha_a);
                else if (p.alpha_a_scope == 2 && row < p.M) aa = __ldg(p.alpha_a + row);
                const uint32_t rbase_off = (uint32_t)(lane * 2 * EPI_COLS);
#pragma unroll 1
                for (int c = 0; c < DQ_TN / 2 / 32; ++c) {
                    float v[32];
                    tmem_ld32(tmem + half * DQ_TN + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * (DQ_TN / 2) + c * 32), v);
                    uint32_t packed[16];
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2)
                        packed[i2] = pack_bf16x2(__fmul_rn(v[2 * i2], aa), __fmul_rn(v[2 * i2 + 1], aa));
                    if (wrow0 < p.M) {
#pragma unroll
                        for (int s2 = 0; s2 < 2; ++s2) {
                            const int64_t col0 = tile.n0 + h * (DQ_TN / 2) + c * 32 + s2 * EPI_COLS;
                            if (col0 < p.N) {
                                const uint32_t buf = ebase + (epi_chunk & 1u) * (uint32_t)EPI_BUF_BYTES;
                                ++epi_chunk;
                                if (lane == 0) bulk_wait_group_read1();
                                __syncwarp();
#pragma unroll
                                for (int j = 0; j < 2; ++j) {
                                    const uint32_t phys = (uint32_t)j ^ ((uint32_t)(lane >> 2) & 1u);
                                    const int pk = s2 * 8 + 4 * j;
                                    st_shared_v4(buf + rbase_off + 16u * phys, packed[pk], packed[pk + 1], packed[pk + 2], packed[pk + 3]);
                                }
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    tma_store_2d(&tmD, (int32_t)col0, (int32_t)wrow0, buf);
                                    bulk_commit_group();
                                }
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader);
        }
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    } else if (warp < DQ_QPROD_WARP) {
        // ------------------------------- converters (both CTAs) -------------------------------
        if constexpr (WG) {
            // B = X (tokens along K): thread ct expands token row t = ct / 4 of the stage, values
            // 32 (ct % 4) .. + 31 of this CTA's 128 B columns, into the MN-major tile (64 B columns per
            // 128-byte row, one row per token, 128-byte swizzle); S is the token's second-level scale.
            const int ct = threadIdx.x - 32 * DQ_CONV_WARP0;
            const int t = ct >> 2, quarter = ct & 3;
            const uint32_t sf_col = (uint32_t)((quarter >> 1) * 512 + (quarter & 1) * 2);
            const uint32_t row_off = (uint32_t)((quarter >> 1) * DQ_MN_ATOM + t * 128);
            int stage = 0, qstage = 0;
            uint32_t phase = 0, qphase = 0;
            bool ok = true;
            for (int64_t tt = pair_id; tt < total_tiles && ok; tt += n_pairs) {
                for (int64_t ks = 0; ks < p.k_stages; ++ks) {
                    if (!warp_wait(bar_qfull + 8 * qstage, qphase, abort_flag, &g_mx_device_status)) { ok = false; break; }
                    if (!warp_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag, &g_mx_device_status)) { ok = false; break; }
                    const int64_t tok = ks * 64 + t;
                    const float S = p.sb2_scope == 1 ? __ldg(p.sb2) : (tok < p.K ? __ldg(p.sb2 + tok) : 0.0f);
                    const uint4 c4 = *reinterpret_cast<const uint4*>(smem + C::SMEM_Q + qstage * C::Q_BYTES + t * 64 + quarter * 16);
                    const uint32_t tb = (uint32_t)(tok & 127);
                    const uint32_t bs2 = *reinterpret_cast<const uint16_t*>(
                        smem + C::SMEM_SF + qstage * C::SF_BYTES + sf_col + (tb & 31) * 16 + ((tb >> 5) & 3) * 4);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_qempty + 8 * qstage);
                    if (++qstage == C::NQ) { qstage = 0; qphase ^= 1; }
                    const uint32_t w[4] = {c4.x, c4.y, c4.z, c4.w};
                    const uint32_t sB = sbase + C::SMEM_B + stage * C::B_BYTES + row_off;
#pragma unroll
                    for (int i2 = 0; i2 < 4; ++i2) {
                        const uint32_t c = (uint32_t)((quarter & 1) * 4 + i2);      // 16-byte chunk of the row
                        const uint32_t bs_h2 = e4m3_to_f16x2_bcast((bs2 >> (8 * (i2 >> 1))) & 0xFFu);
                        const uint4 o = dq_word(w[i2], bs_h2, S);
                        st_shared_v4(sB + 16u * (c ^ (uint32_t)(t & 7)), o.x, o.y, o.z, o.w);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(leader ? bar_full + 8 * stage : bar_bconv + 8 * stage);
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && lane == 0) *abort_flag = 1;
        } else {
            // thread ct: B row r of this CTA's half, chunks [part * DQ_CONV_CHUNKS, +DQ_CONV_CHUNKS) of its 8
            const int ct = threadIdx.x - 32 * DQ_CONV_WARP0;
            const int r = ct / (8 / DQ_CONV_CHUNKS), part = ct % (8 / DQ_CONV_CHUNKS);
            const uint32_t row_off = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128);
            const uint32_t sf_off = (uint32_t)((r & 31) * 16 + ((r >> 5) & 3) * 4);
            int stage = 0, qstage = 0;
            uint32_t phase = 0, qphase = 0;
            bool ok = true;
            for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs) {
                const PairTile tile = dq_tile(p, t, rank);
                const int64_t brow = tile.n0 + 128 * (int64_t)rank + r;
                float S = 0.0f;
                if (p.sb2_scope == 1) S = __ldg(p.sb2);
                else if (brow < p.N) S = __ldg(p.sb2 + brow);
                for (int64_t ks = 0; ks < p.k_stages; ++ks) {
                    if (!warp_wait(bar_qfull + 8 * qstage, qphase, abort_flag, &g_mx_device_status)) { ok = false; break; }
                    if (!warp_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag, &g_mx_device_status)) { ok = false; break; }
                    const uint8_t* qsrc = smem + C::SMEM_Q + qstage * C::Q_BYTES + r * 32 + part * 4 * DQ_CONV_CHUNKS;
                    uint32_t w[DQ_CONV_CHUNKS];
                    if constexpr (DQ_CONV_CHUNKS >= 4) {
#pragma unroll
                        for (int i = 0; i < DQ_CONV_CHUNKS; i += 4) {
                            const uint4 c4 = *reinterpret_cast<const uint4*>(qsrc + 4 * i);
                            w[i] = c4.x; w[i + 1] = c4.y; w[i + 2] = c4.z; w[i + 3] = c4.w;
                        }
                    } else {
                        const uint2 c2 = *reinterpret_cast<const uint2*>(qsrc);
                        w[0] = c2.x; w[1] = c2.y;
                    }
                    const uint32_t sc = *reinterpret_cast<const uint32_t*>(smem + C::SMEM_SF + qstage * C::SF_BYTES + sf_off);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_qempty + 8 * qstage);            // codes slot read
                    if (++qstage == C::NQ) { qstage = 0; qphase ^= 1; }
                    const uint32_t sB = sbase + C::SMEM_B + stage * C::B_BYTES + row_off;
#pragma unroll
                    for (int i = 0; i < DQ_CONV_CHUNKS; ++i) {
                        // chunk ci = values 8 ci .. 8 ci + 7 of the stage, block ci / 2 of the row's four
                        const int ci = part * DQ_CONV_CHUNKS + i;
                        const uint32_t bs_h2 = e4m3_to_f16x2_bcast((sc >> (8 * (ci >> 1))) & 0xFFu);
                        const uint4 o = dq_word(w[i], bs_h2, S);
                        st_shared_v4(sB + 16u * ((uint32_t)ci ^ (uint32_t)(r & 7)), o.x, o.y, o.z, o.w);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(leader ? bar_full + 8 * stage : bar_bconv + 8 * stage);
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && lane == 0) *abort_flag = 1;
        }
    } else {
        // ------------------------------- codes producer (both CTAs) -------------------------------
        // codes and scale atom of this CTA's 128 B rows, up to NQ stages ahead of the converters
        int qstage = 0;
        uint32_t qphase = 0;
        bool ok = true;
        for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs) {
            const PairTile tile = dq_tile(p, t, rank);
            const int64_t brow = tile.n0 + 128 * (int64_t)rank;
            const int64_t band = brow / 128;
            for (int64_t ks = 0; ks < p.k_stages; ++ks) {
                if (!warp_wait(bar_qempty + 8 * qstage, qphase ^ 1, abort_flag, &g_mx_device_status)) { ok = false; break; }
                if (elect_one()) {
                    const uint32_t qb = bar_qfull + 8 * qstage;
                    mbar_arrive_expect_tx(qb, C::Q_TX);
                    if constexpr (WG) {
                        // 64 tokens x this CTA's 128 B columns of X's codes; the two scale atoms of those
                        // columns in the tokens' 128-row band
                        tma_load_2d(sbase + C::SMEM_Q + qstage * C::Q_BYTES, &tmQ, (int32_t)(brow / 2), (int32_t)(ks * 64), qb);
                        tma_load_2d(sbase + C::SMEM_SF + qstage * C::SF_BYTES, &tmSB, 0,
                                    (int32_t)((((ks * 64) / 128) * p.nct + brow / 64) * 2), qb);
                    } else {
                        tma_load_2d(sbase + C::SMEM_Q + qstage * C::Q_BYTES, &tmQ, (int32_t)(ks * 32), (int32_t)brow, qb);
                        tma_load_2d(sbase + C::SMEM_SF + qstage * C::SF_BYTES, &tmSB, 0, (int32_t)((band * p.nct + ks) * 2), qb);
                    }
                }
                __syncwarp();
                if (++qstage == C::NQ) { qstage = 0; qphase ^= 1; }
            }
        }
        if (!ok && lane == 0) *abort_flag = 1;
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {}
    }
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
}

// ---------------------------------------------------------------------------------------------
// Blockwise FP8 GEMM with FP32 scales (NeMo RL FP8 page, "FP8 nas camadas lineares": the DeepSeek-V3
// recipe, [1, 128] activation / gradient tiles and [128, 128] weight blocks with FP32 scales; E2E page
// Table 1: on SM100 the tensor cores take power-of-two block scales natively, FP32 ones are applied
// around them):
//   D[m, n] = BF16( sum_kb sa[m, kb] * sb[n / 128, kb] * P_kb[m, n] ),   P_kb = sum_{k in kb} A[m, k] B[n, k]
// and, for the weight gradient (both operands contracted over tokens, so both in [1, 128] tiles along K,
// BROW = true), the same with one B scale per B row:  sb[n, kb] in place of sb[n / 128, kb].
// Each 128-deep K block's P_kb comes from plain E4M3 pair MMAs (kind::f8f6f4, FP32 accumulation) into
// one of four TMEM buffers (4 x 128 columns); the 8 epilogue warps promote it into FP32 register
// accumulators with the block's scale product (packed two-lane FP32 multiply-adds) while the tensor
// core fills the other buffers, and write the tile once all K blocks are in.  With per-row B scales each
// epilogue warp stages the scales of its 64 columns for four K blocks at a time in a slot of its own in
// shared memory (transposed, so every lane reads them as broadcasts), loading the next four ahead.
// Warp 0 loads A and B by TMA (as the block-scaled kernel, without scale atoms); warp 1 of the even CTA
// issues the MMAs; warp 1 of the odd CTA forwards its epilogue's "buffer read" to the even CTA as a
// 16-byte bulk copy.
// ---------------------------------------------------------------------------------------------
struct BwParams {
    const float* sa; const float* sb;       // sa [M, K/128]; sb [ceil(N/128), K/128], or [N, K/128] (per-row B)
    int64_t M, N, K, kb_n, nb_n;
    uint16_t* d; int64_t ldd;
    int64_t m_tiles, n_tiles, total_tiles;
};

// Issue a load of 16 TMEM columns of this warp's 32 lanes; the registers are valid only after
// tmem_wait_ld on them.
__device__ __forceinline__ void tmem_ld_issue(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr) : "memory");
}
// Wait for this thread's TMEM loads.  The registers pass through the statement, so no use of them
// can be scheduled above the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
        :: "memory");
}

template <int TN, bool BROW>
struct BwCfg {
    static constexpr int NP = TMEM_COLS / TN;              // partial-product buffers in TMEM
    static constexpr int NST = TN == 256 ? 6 : 8;
    static constexpr int A_BYTES = 128 * BKB;              // 128 rows x 128 E4M3
    static constexpr int B_BYTES = (TN / 2) * BKB;         // this CTA's half of the TN B rows
    static constexpr uint32_t STAGE_TX = 2u * (A_BYTES + B_BYTES);
    static constexpr int SMEM_A = 0;
    static constexpr int SMEM_B = SMEM_A + NST * A_BYTES;
    static constexpr int SMEM_EPI = SMEM_B + NST * B_BYTES;
    static constexpr int SMEM_BAR = SMEM_EPI + EPI_WARPS * 2 * EPI_BUF_BYTES;
    static constexpr int SMEM_MISC = SMEM_BAR + 8 * (2 * NST + 3 * NP + 1);
    static constexpr int SMEM_SIGNAL = (SMEM_MISC + 16 + 15) / 16 * 16;
    // per-row B scales: one slot per epilogue warp of 4 K blocks x TN/2 columns (FP32)
    static constexpr int SB_SLOT_FLOATS = 2 * 4 * (TN / 2);   // two groups of four K blocks
    static constexpr int SMEM_SB = SMEM_SIGNAL + 16;
    static constexpr int SMEM_ALLOC = SMEM_SB + (BROW ? EPI_WARPS * SB_SLOT_FLOATS * 4 : 0) + 1024;
    static_assert(SMEM_B % 1024 == 0 && SMEM_EPI % 1024 == 0 && SMEM_SB % 16 == 0, "alignment");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// kind::f8f6f4 without block scaling: D FP32 (bits 4-5 = 1), A and B E4M3 (format 0), K-major.
template <int MMA_M, int MMA_N>
__device__ __forceinline__ uint32_t make_idesc_e4m3() {
    return (1u << 4) | ((uint32_t)(MMA_N >> 3) << 17) | ((uint32_t)(MMA_M >> 4) << 24);
}

__device__ __forceinline__ void tc2_mma_e4m3(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
}

// 4-byte asynchronous global -> shared copy; src_bytes = 0 stores a zero instead (the source is not read).
__device__ __forceinline__ void cp_async_f32(uint32_t dst, const float* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Promotion of one CW-column chunk of a K block's partial product into the FP32 accumulators:
//   acc[c] += P[c] * scale                 (forward forms: one factor per row and K block)
//   acc[c] += P[c] * (scale * sb[c])       (per-row B: the column's scale from the warp's slot at srow)
// as packed two-lane FP32 operations (IEEE round-to-nearest per lane).
template <bool BROW, int CW>
__device__ __forceinline__ void promote_chunk(uint64_t* acc, const uint32_t (&v)[CW], uint64_t scale2, uint32_t srow) {
#pragma unroll
    for (int i = 0; i < CW / 4; ++i) {
        const uint64_t p0 = f2_pack(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]));
        const uint64_t p1 = f2_pack(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        if (BROW) {
            uint64_t s01, s23;                                  // column scales 4i..4i+3 (broadcast)
            asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(s01), "=l"(s23) : "r"(srow + (uint32_t)(16 * i)));
            acc[2 * i] = f2_fma(p0, f2_mul(s01, scale2), acc[2 * i]);
            acc[2 * i + 1] = f2_fma(p1, f2_mul(s23, scale2), acc[2 * i + 1]);
        } else {
            acc[2 * i] = f2_fma(p0, scale2, acc[2 * i]);
            acc[2 * i + 1] = f2_fma(p1, scale2, acc[2 * i + 1]);
        }
    }
}

template <int TN, bool BROW>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
fp8bw_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmD, const BwParams p) {
    using C = BwCfg<TN, BROW>;
    constexpr int NST = C::NST;
    constexpr int NP = C::NP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + C::SMEM_BAR;            // NST (even CTA): both CTAs' A and B bytes
    const uint32_t bar_empty = bar_full + 8 * NST;            // NST (each CTA)
    const uint32_t bar_pfull = bar_empty + 8 * NST;           // NP (each CTA): a K block's partial product is in TMEM
    const uint32_t bar_pempty = bar_pfull + 8 * NP;           // NP (even CTA): both epilogues have read it
    const uint32_t bar_pempty_odd = bar_pempty + 8 * NP;      // NP (odd CTA): its epilogue has read it
    const uint32_t bar_done = bar_pempty_odd + 8 * NP;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SMEM_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::SMEM_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < NP; ++b) {
            mbar_init(bar_pfull + 8 * b, 1);
            mbar_init(bar_pempty + 8 * b, EPI_WARPS);             // one arrival also expects the odd CTA's copy
            mbar_init(bar_pempty_odd + 8 * b, EPI_WARPS);
        }
        mbar_init(bar_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmA) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmB) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(&tmD) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int64_t total_tiles = p.total_tiles;
    const int64_t pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    Params tp{};
    tp.M = p.M; tp.N = p.N; tp.m_tiles = p.m_tiles; tp.n_tiles = p.n_tiles; tp.d = p.d; tp.ldd = p.ldd;

    if (warp == 0) {
        // ------------------------------- producer (both CTAs) -------------------------------
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs) {
            const PairTile tile = pair_dense_tile<TN>(tp, t, rank);
            const int64_t brow = tile.n0 + (TN / 2) * (int64_t)rank;
            for (int64_t kb = 0; kb < p.kb_n; ++kb) {
                if (!warp_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag, &g_mx_device_status)) { ok = false; break; }
                if (elect_one()) {
                    const uint32_t fb = map_to_cta(bar_full + 8 * stage, 0);
                    if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, C::STAGE_TX);
                    tma_load_2d_pair(sbase + C::SMEM_A + stage * C::A_BYTES, &tmA, (int32_t)(kb * BKB), (int32_t)tile.row0, fb);
                    tma_load_2d_pair(sbase + C::SMEM_B + stage * C::B_BYTES, &tmB, (int32_t)(kb * BKB), (int32_t)brow, fb);
                }
                __syncwarp();
                if (++stage == NST) { stage = 0; phase ^= 1; }
            }
        }
        if (!ok && lane == 0) *abort_flag = 1;
    } else if (warp == 1) {
        if (leader) {
            // ------------------------------- MMA (even CTA) -------------------------------
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, issued_any = false;
            int64_t g = 0;                                   // K blocks issued so far: buffer g % NP
            for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs) {
                for (int64_t kb = 0; kb < p.kb_n; ++kb, ++g) {
                    const uint32_t pb = (uint32_t)(g % NP), use = (uint32_t)(g / NP);
                    if (!warp_wait(bar_pempty + 8 * pb, (use & 1u) ^ 1u, abort_flag, &g_mx_device_status)) { ok = false; break; }
                    if (!warp_wait(bar_full + 8 * stage, phase, abort_flag, &g_mx_device_status)) { ok = false; break; }
                    tc_fence_after();
                    if (elect_one()) {
                        const uint32_t sA = sbase + C::SMEM_A + stage * C::A_BYTES;
                        const uint32_t sB = sbase + C::SMEM_B + stage * C::B_BYTES;
#pragma unroll
                        for (int j = 0; j < BKB / 32; ++j)
                            tc2_mma_e4m3(tmem + pb * TN, desc_sw128(sA + 32 * j), desc_sw128(sB + 32 * j),
                                         make_idesc_e4m3<2 * BM, TN>(), j > 0 ? 1u : 0u);
                        tc2_commit_mc(bar_empty + 8 * stage, (uint16_t)3);
                        tc2_commit_mc(bar_pfull + 8 * pb, (uint16_t)3);
                    }
                    __syncwarp();
                    issued_any = true;
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
            }
            // the last buffer releases (the odd CTA's arrive as copies) complete before either CTA leaves
            for (int b = 0; b < NP && ok; ++b) {
                const int64_t uses = (g - b + NP - 1) / NP;
                if (uses > 0 && !warp_wait(bar_pempty + 8 * b, (uint32_t)((uses - 1) & 1), abort_flag, &g_mx_device_status))
                    ok = false;
            }
            if (issued_any) {
                if (elect_one()) {
                    tc2_commit_mc(bar_done, (uint16_t)1);
                    const unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(bar_done, 0) && globaltimer() - t0 < WAIT_LIMIT_NS) {}
                }
                __syncwarp();
            }
        } else {
            // odd CTA: forward each "partial buffer read" of this CTA's epilogue to the even CTA
            const uint32_t pempty_leader = map_to_cta(bar_pempty, 0);
            const uint32_t sig_dst = map_to_cta(sbase + C::SMEM_SIGNAL, 0);
            bool ok = true;
            int64_t g = 0;
            for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs) {
                for (int64_t kb = 0; kb < p.kb_n; ++kb, ++g) {
                    const uint32_t pb = (uint32_t)(g % NP), use = (uint32_t)(g / NP);
                    if (!warp_wait(bar_pempty_odd + 8 * pb, use & 1u, abort_flag, &g_mx_device_status)) { ok = false; break; }
                    if (lane == 0) bulk_signal_copy(sig_dst, sbase + C::SMEM_SIGNAL, 16, pempty_leader + 8 * pb);
                    __syncwarp();
                }
            }
            if (!ok && lane == 0) *abort_flag = 1;
        }
    } else {
        // ------------------------------- promotion + epilogue (both CTAs) -------------------------------
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const uint32_t ebase = sbase + C::SMEM_EPI + (uint32_t)((warp - 2) * 2 * EPI_BUF_BYTES);
        const uint32_t my_pempty = leader ? bar_pempty : bar_pempty_odd;
        // per-row B scales: this warp's slot, [4 K blocks][TN/2 columns]
        float* sb_slot = reinterpret_cast<float*>(smem + C::SMEM_SB) + (warp - 2) * C::SB_SLOT_FLOATS;
        const uint32_t sb_slot_s = smem_u32(sb_slot);
        uint32_t epi_chunk = 0;
        int64_t g = 0;
        bool ok = true;
        const int32_t kb_n32 = (int32_t)p.kb_n;
        for (int64_t t = pair_id; t < total_tiles && ok; t += n_pairs) {
            const PairTile tile = pair_dense_tile<TN>(tp, t, rank);
            const int64_t row = tile.row0 + q * 32 + lane;
            const int64_t col0 = tile.n0 + h * (TN / 2);            // first output column of this warp
            const int64_t nblk = col0 / 128;
            const bool row_ok = row < p.M;
            const bool blk_ok = BROW || nblk < p.nb_n;
            const float* sa_row = p.sa + (row_ok ? row : 0) * p.kb_n;
            const float* sb_blk = p.sb + (!BROW && blk_ok ? nblk : 0) * p.kb_n;
            // Per-row B: lane l copies the scales of its columns col0 + l + 32 c (zero past N or past K) for four
            // K blocks at a time straight into the warp's slot, transposed, two groups ahead by asynchronous
            // copies (slot buffer = group parity), and its row scales sa are loaded a group ahead; the forward
            // forms read sa and the block scales per K block (each measured faster than the other way).
            constexpr int SBC = TN / 64;
            const float* sb_lane = p.sb + (BROW ? (col0 + lane) * p.kb_n : 0);
            uint32_t sb_okm = 0;                                        // bit c: column c of this lane exists
#pragma unroll
            for (int c = 0; c < SBC; ++c) sb_okm |= (BROW && col0 + lane + 32 * c < p.N) ? (1u << c) : 0u;
            auto stage_group = [&](int32_t grp) {
                const uint32_t dst = sb_slot_s + (uint32_t)((grp & 1) * 4 * (TN / 2) * 4);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int32_t k = 4 * grp + j;
#pragma unroll
                    for (int c = 0; c < SBC; ++c) {
                        const bool in = ((sb_okm >> c) & 1u) && k < kb_n32;
                        cp_async_f32(dst + (uint32_t)((j * (TN / 2) + 32 * c + lane) * 4),
                                     in ? sb_lane + (int64_t)32 * c * kb_n32 + k : p.sb, in ? 4u : 0u);
                    }
                }
                cp_async_commit();
            };
            if (BROW) {
                cp_async_wait0();                      // the previous tile's copies have landed
                __syncwarp();
                stage_group(0);
                stage_group(1);
            }
            uint32_t packed[TN / 4];                       // the tile's BF16 results, this warp's slice
            if constexpr (BROW) {
            // Per-row B: software pipeline over 16-column chunks of each K block: one TMEM load is in flight
            // while the previous chunk is promoted (two packed operations per column pair), the first chunk
            // of kb + 1 behind the last of kb.
            constexpr int CW = 16;                         // measured faster than 32-column chunks (1.07 / 1.17 ms)
            constexpr int NCH = (TN / 2) / CW;
            static_assert(NCH % 2 == 0, "chunk parity alternates the two register sets");
            uint64_t acc[TN / 4];
#pragma unroll
            for (int i = 0; i < TN / 4; ++i) acc[i] = 0ull;
            const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * (TN / 2));
            uint32_t va[CW], vb[CW];
            float sa_next[4], sa_cur[4];                   // row scales of four K blocks, a group ahead
#pragma unroll
            for (int j = 0; j < 4; ++j) sa_next[j] = row_ok && j < kb_n32 ? __ldg(sa_row + j) : 0.0f;
            if (kb_n32 > 0) {
                const uint32_t pb0 = (uint32_t)(g % NP), use0 = (uint32_t)(g / NP);
                if (!mbar_wait(bar_pfull + 8 * pb0, use0 & 1u, abort_flag, &g_mx_device_status)) { ok = false; break; }
                tc_fence_after();
                tmem_ld_issue(lane_base + pb0 * TN, va);
                tmem_wait_ld(va);
            }
            for (int32_t kb = 0; kb < kb_n32 && ok; ++kb, ++g) {
                const uint32_t pb = (uint32_t)(g % NP);
                const int32_t j4 = kb & 3;
                if (j4 == 0) {
                    // a new group of four K blocks: its row scales become current (the next group's are
                    // fetched), and its column scales' copies are waited for
#pragma unroll
                    for (int j = 0; j < 4; ++j) sa_cur[j] = sa_next[j];
#pragma unroll
                    for (int j = 0; j < 4; ++j) sa_next[j] = row_ok && kb + 4 + j < kb_n32 ? __ldg(sa_row + kb + 4 + j) : 0.0f;
                    cp_async_wait1();                      // all but the newest group: this one has landed
                    __syncwarp();
                }
                const float scale = j4 == 0 ? sa_cur[0] : j4 == 1 ? sa_cur[1] : j4 == 2 ? sa_cur[2] : sa_cur[3];
                const uint64_t scale2 = f2_pack(scale, scale);
                const uint32_t srow = sb_slot_s + (uint32_t)((((kb >> 2) & 1) * 4 + j4) * (TN / 2) * 4);
                const bool more = kb + 1 < kb_n32;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    uint32_t (&cur)[CW] = (c & 1) ? vb : va;
                    uint32_t (&nxt)[CW] = (c & 1) ? va : vb;
                    if (c + 1 < NCH) {
                        tmem_ld_issue(lane_base + pb * TN + (uint32_t)((c + 1) * CW), nxt);
                        promote_chunk<true, CW>(acc + c * (CW / 2), cur, scale2, srow + (uint32_t)(c * CW * 4));
                        tmem_wait_ld(nxt);
                        if (c + 2 == NCH) {
                            // the whole K block is in registers: hand the buffer back
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) {
                                if (leader && warp == 2) mbar_arrive_expect_tx(my_pempty + 8 * pb, 16);
                                else mbar_arrive(my_pempty + 8 * pb);
                            }
                        }
                    } else {
                        if (more) {
                            const uint32_t pn = (uint32_t)((g + 1) % NP), usen = (uint32_t)((g + 1) / NP);
                            if (!mbar_wait(bar_pfull + 8 * pn, usen & 1u, abort_flag, &g_mx_device_status)) ok = false;
                            tc_fence_after();
                            if (ok) tmem_ld_issue(lane_base + pn * TN, nxt);          // chunk 0 of kb + 1
                        }
                        promote_chunk<true, CW>(acc + c * (CW / 2), cur, scale2, srow + (uint32_t)(c * CW * 4));
                        if (more && ok) tmem_wait_ld(nxt);
                    }
                }
                if (j4 == 3) {
                    // the group's slot buffer is read: refill it with the group after next
                    __syncwarp();
                    stage_group((kb >> 2) + 2);
                }
            }
#pragma unroll
            for (int i = 0; i < TN / 4; ++i) {
                float lo, hi;
                f2_unpack(acc[i], lo, hi);
                packed[i] = pack_bf16x2(lo, hi);
            }
            } else {
            // Forward forms: promotion one K block at a time, the partial product's 32-column chunks loaded
            // from TMEM and accumulated with the block's factor (scalar FP32 multiply-adds: measured faster
            // here than the packed form), then the buffer handed back.
            float accf[TN / 2];
#pragma unroll
            for (int i = 0; i < TN / 2; ++i) accf[i] = 0.0f;
            for (int32_t kb = 0; kb < kb_n32; ++kb, ++g) {
                const uint32_t pb = (uint32_t)(g % NP), use = (uint32_t)(g / NP);
                const float scale = (row_ok && blk_ok) ? __fmul_rn(__ldg(sa_row + kb), __ldg(sb_blk + kb)) : 0.0f;
                if (!mbar_wait(bar_pfull + 8 * pb, use & 1u, abort_flag, &g_mx_device_status)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < TN / 2 / 32; ++c) {
                    float v[32];
                    tmem_ld32(tmem + pb * TN + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * (TN / 2) + c * 32), v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) accf[c * 32 + i] = __fmaf_rn(v[i], scale, accf[c * 32 + i]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (leader && warp == 2) mbar_arrive_expect_tx(my_pempty + 8 * pb, 16);
                    else mbar_arrive(my_pempty + 8 * pb);
                }
            }
#pragma unroll
            for (int i = 0; i < TN / 4; ++i) packed[i] = pack_bf16x2(accf[2 * i], accf[2 * i + 1]);
            }
            if (!ok) break;
            epilogue_store<TN, false, 2, EPI_COLS>(tp, &tmD, q, h, lane, tile.row0, tile.row_end, tile.n0, ebase, epi_chunk, packed);
        }
        if (BROW) cp_async_wait0();                   // no copy into this warp's slot outlives the CTA
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {}
    }
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
}

// ---------------------------------------------------------------------------------------------
// Watchdog self-test: one cluster of two CTAs set up as the pair GEMMs are (mbarriers initialised
// for the cluster, the pair's TMEM allocation, a CTA-local abort flag), in which every role waits on
// a barrier that nothing ever arrives on, with the caller's limit instead of the kernels' 2 s.  The
// first wait to give up sets the timeout bit of this file's status word and the CTA's abort flag;
// the other roles see the flag and leave; then the CTAs take the GEMMs' exit path (CTA barrier,
// cluster barrier, TMEM release).  No copy and no MMA is ever issued, so nothing is in flight at exit.
// ---------------------------------------------------------------------------------------------
constexpr uint32_t WATCHDOG_TMEM_COLS = 32;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
watchdog_selftest_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bars[3];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_s;
    volatile int* abort_flag = &abort_s;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&bars[i]), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&tmem_slot)), "r"(WATCHDOG_TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // phase 0 of each barrier never completes: every wait below ends by its limit or by the abort flag
    if (warp == 0) {
        warp_wait(smem_u32(&bars[0]), 0, abort_flag, &g_mx_device_status, limit_ns);        // producer role
    } else if (warp == 1) {
        warp_wait(smem_u32(&bars[1]), 0, abort_flag, &g_mx_device_status, limit_ns);        // MMA role
    } else {
        mbar_wait_backoff(smem_u32(&bars[2]), 0, abort_flag, &g_mx_device_status, limit_ns);  // epilogue role
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(WATCHDOG_TMEM_COLS) : "memory");
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
bool make_map(CUtensorMap* map, const uint8_t* base, int64_t k_bytes, int64_t rows, uint32_t box_rows) {
    return encode_tensor_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, (uint64_t)k_bytes, (uint64_t)rows,
                                (uint64_t)k_bytes, (uint32_t)BKB, box_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// Output map: BF16 [rows, N] with row pitch ldd, box of `box_cols` x 32 rows, swizzled to match the
// epilogue's staging layout.
bool make_out_map(CUtensorMap* map, uint16_t* d, int64_t rows, int64_t N, int64_t ldd, uint32_t box_cols) {
    const CUtensorMapSwizzle sw = box_cols * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : box_cols * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    return encode_tensor_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, d, (uint64_t)N, (uint64_t)rows, (uint64_t)(ldd * 2),
                                box_cols, 32, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// Scale tensor viewed as rows of 256 bytes (two rows per 512-byte atom), box of `atoms` atoms.
bool make_sf_map(CUtensorMap* map, const uint8_t* base, int64_t bytes, uint32_t atoms) {
    return encode_tensor_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 256, (uint64_t)(bytes / 256), 256, 256,
                                2 * atoms, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

template <int FMT, bool GROUPED, bool COL_ALPHA, int TN, int EV = 0>
cudaError_t launch_pair_impl(const GemmArgs& a, int num_sms, cudaStream_t stream) {
    using C = PairCfg<FMT, GROUPED, TN, EV>;
    static PerDevice setup;                 // attributes, and the CTA pairs that fit on the GPU at once
    int resident_pairs = 0;
    const cudaError_t attr_err = per_device_once(setup, resident_pairs, [num_sms](int& rp) -> cudaError_t {
        auto kern = bs_gemm_pair_kernel<FMT, GROUPED, COL_ALPHA, TN, EV>;
        // grouped launches size their tables by G: allow up to the per-block limit
        const int max_alloc = GROUPED ? C::SMEM_LIMIT : C::SMEM_ALLOC;
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_alloc);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(num_sms & ~1));
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = max_alloc;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2; attr[0].val.clusterDim.y = 1; attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr; cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = num_sms / 2;
        }
        rp = n;
        return cudaSuccess;
    });
    if (attr_err != cudaSuccess) return attr_err;

    const int64_t k_bytes = FMT == 0 ? a.K : a.K / 2;
    const int block = FMT == 0 ? 32 : 16;
    // scale tensor sizes as the API defines them (grouped A: every group padded to 128-row bands)
    const int64_t sa_bytes = GROUPED ? host_scale_bytes(a.M + 127 * a.G, a.K, block) : host_scale_bytes(a.M, a.K, block);
    const int64_t sb_group_bytes = host_scale_bytes(a.N, a.K, block);
    const int64_t sb_bytes = (GROUPED ? a.G : 1) * sb_group_bytes;
    CUtensorMap tmA, tmB, tmSA, tmSB, tmD;
    if (!make_map(&tmA, a.a, k_bytes, a.M, 128)) return cudaErrorInvalidValue;
    if (!make_map(&tmB, a.b, k_bytes, GROUPED ? a.G * a.N : a.N, (uint32_t)C::B_BOX)) return cudaErrorInvalidValue;
    if (!make_sf_map(&tmSA, a.sa, sa_bytes, (uint32_t)C::SF_ATOMS_A)) return cudaErrorInvalidValue;
    if (!make_sf_map(&tmSB, a.sb, sb_bytes, (uint32_t)C::SF_ATOMS_A)) return cudaErrorInvalidValue;   // one band per load
    if (!make_out_map(&tmD, a.d, a.M, a.N, a.ldd, (uint32_t)C::EPI_C)) return cudaErrorInvalidValue;

    Params p{};
    p.sa = a.sa; p.sb = a.sb;
    p.alpha_a = a.alpha_a; p.alpha_a_scope = a.alpha_a_scope;
    p.alpha_b = a.alpha_b; p.alpha_b_scope = a.alpha_b_scope;
    p.M = a.M; p.N = a.N; p.K = a.K; p.d = a.d; p.ldd = a.ldd;
    p.G = a.G; p.group_offsets = a.group_offsets;
    p.m_tiles = (a.M + 2 * BM - 1) / (2 * BM);        // pair rows (256)
    p.n_tiles = (a.N + TN - 1) / TN;
    p.k_stages = k_bytes / BKB;
    p.nct = (a.K / block + 3) / 4;
    p.sb_group_bytes = sb_group_bytes;
    p.total_tiles = p.m_tiles * p.n_tiles;
    const int64_t tiles_bound = GROUPED ? (p.m_tiles + a.G) * p.n_tiles : p.total_tiles;
    // a persistent grid: only as many pairs as can be resident together (an odd SM left in a GPC
    // cannot host half a cluster)
    const int64_t pairs = max64(1, min64(tiles_bound, (int64_t)min(resident_pairs, num_sms / 2)));
    if (GROUPED && a.G > C::MAX_G) return cudaErrorInvalidValue;
    bs_gemm_pair_kernel<FMT, GROUPED, COL_ALPHA, TN, EV><<<(unsigned)(2 * pairs), NUM_THREADS, C::smem_alloc(a.G), stream>>>(
        tmA, tmB, tmSA, tmSB, tmD, p);
    return cudaGetLastError();
}

template <bool WG>
cudaError_t launch_dq_impl(const DqGemmArgs& a, int num_sms, cudaStream_t stream) {
    using C = DqCfg<WG>;
    static PerDevice setup;                 // attributes, and the CTA pairs that fit on the GPU at once
    int resident_pairs = 0;
    const cudaError_t attr_err = per_device_once(setup, resident_pairs, [num_sms](int& rp) -> cudaError_t {
        const cudaError_t e = cudaFuncSetAttribute(dq_gemm_pair_kernel<WG>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(num_sms & ~1));
        cfg.blockDim = dim3(DQ_THREADS);
        cfg.dynamicSmemBytes = C::SMEM_ALLOC;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2; attr[0].val.clusterDim.y = 1; attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr; cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, dq_gemm_pair_kernel<WG>, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = num_sms / 2;
        }
        rp = n;
        return cudaSuccess;
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tmA, tmQ, tmSB, tmD;
    if constexpr (WG) {
        // A = dY [K = T, M = O] read in 64 x 64 boxes (MN-major); B codes = X [K = T, N/2] in boxes of
        // 64 tokens x 64 bytes; X's scales (T, N, 16) in two-atom boxes
        if (!encode_tensor_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.a, (uint64_t)a.M, (uint64_t)a.K,
                                  (uint64_t)(a.M * 2), 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
            return cudaErrorInvalidValue;
        if (!encode_tensor_map_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.qb, (uint64_t)(a.N / 2), (uint64_t)a.K,
                                  (uint64_t)(a.N / 2), 64, 64, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
            return cudaErrorInvalidValue;
        if (!make_sf_map(&tmSB, a.sb, host_scale_bytes(a.K, a.N, 16), 2)) return cudaErrorInvalidValue;
    } else {
        if (!make_map(&tmA, reinterpret_cast<const uint8_t*>(a.a), a.K * 2, a.M, 128)) return cudaErrorInvalidValue;
        if (!encode_tensor_map_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.qb, (uint64_t)(a.K / 2), (uint64_t)a.N,
                                  (uint64_t)(a.K / 2), 32, 128, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
            return cudaErrorInvalidValue;
        if (!make_sf_map(&tmSB, a.sb, host_scale_bytes(a.N, a.K, 16), 1)) return cudaErrorInvalidValue;
    }
    if (!make_out_map(&tmD, a.d, a.M, a.N, a.ldd, (uint32_t)EPI_COLS)) return cudaErrorInvalidValue;
    DqParams p{};
    p.alpha_a = a.alpha_a; p.alpha_a_scope = a.alpha_a_scope;
    p.sb2 = a.sb2; p.sb2_scope = a.sb2_scope;
    p.M = a.M; p.N = a.N; p.K = a.K; p.d = a.d; p.ldd = a.ldd;
    p.m_tiles = (a.M + 511) / 512;
    p.n_tiles = (a.N + DQ_TN - 1) / DQ_TN;
    p.k_stages = a.K / 64;
    p.nct = WG ? (a.N / 16 + 3) / 4 : (a.K / 16 + 3) / 4;
    p.total_tiles = p.m_tiles * p.n_tiles;
    const int64_t pairs = max64(1, min64(p.total_tiles, (int64_t)min(resident_pairs, num_sms / 2)));
    dq_gemm_pair_kernel<WG><<<(unsigned)(2 * pairs), DQ_THREADS, C::SMEM_ALLOC, stream>>>(tmA, tmQ, tmSB, tmD, p);
    return cudaGetLastError();
}


template <int TN, bool BROW>
cudaError_t launch_bw_impl(const BwGemmArgs& a, int num_sms, cudaStream_t stream) {
    using C = BwCfg<TN, BROW>;
    static PerDevice setup;                 // attributes, and the CTA pairs that fit on the GPU at once
    int resident_pairs = 0;
    const cudaError_t attr_err = per_device_once(setup, resident_pairs, [num_sms](int& rp) -> cudaError_t {
        const cudaError_t e = cudaFuncSetAttribute(fp8bw_gemm_pair_kernel<TN, BROW>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(num_sms & ~1));
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = C::SMEM_ALLOC;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2; attr[0].val.clusterDim.y = 1; attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr; cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, fp8bw_gemm_pair_kernel<TN, BROW>, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = num_sms / 2;
        }
        rp = n;
        return cudaSuccess;
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tmA, tmB, tmD;
    if (!make_map(&tmA, a.a, a.K, a.M, 128)) return cudaErrorInvalidValue;
    if (!make_map(&tmB, a.b, a.K, a.N, TN / 2)) return cudaErrorInvalidValue;
    if (!make_out_map(&tmD, a.d, a.M, a.N, a.ldd, (uint32_t)EPI_COLS)) return cudaErrorInvalidValue;
    BwParams p{};
    p.sa = a.sa; p.sb = a.sb;
    p.M = a.M; p.N = a.N; p.K = a.K; p.kb_n = a.K / 128; p.nb_n = (a.N + 127) / 128;
    p.d = a.d; p.ldd = a.ldd;
    p.m_tiles = (a.M + 2 * BM - 1) / (2 * BM);
    p.n_tiles = (a.N + TN - 1) / TN;
    p.total_tiles = p.m_tiles * p.n_tiles;
    const int64_t pairs = max64(1, min64(p.total_tiles, (int64_t)min(resident_pairs, num_sms / 2)));
    fp8bw_gemm_pair_kernel<TN, BROW><<<(unsigned)(2 * pairs), NUM_THREADS, C::SMEM_ALLOC, stream>>>(tmA, tmB, tmD, p);
    return cudaGetLastError();
}

}  // namespace


namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}
}  // namespace

bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t outer,
                          uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle,
                          CUtensorMapL2promotion promo) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Dense MXFP8 tile width.  A 256 x 384 tile loads 16 % fewer operand bytes per MMA than a 256 x 256
// one (each A row serves 384 columns instead of 256) and measured 3-5 % faster per tile column on the
// Qwen3-8B MLP shapes, but it wastes the padding of a ragged last column tile and fills the CTA pairs
// in coarser waves.  Estimate each width's time as (waves of tiles over the pairs) x (tile width),
// with the wide tile's rate 4 % better, and take the smaller: FPROP 8192 x 12288 x 4096 and WGRAD
// 12288 x 4096 x 8192 take 384 columns, DGRAD 8192 x 4096 x 12288 and small GEMMs 256.
static bool wide_mxfp8_tiles(const GemmArgs& a, int num_sms) {
    const int64_t pairs = max64(1, num_sms / 2);
    const int64_t m_tiles = (a.M + 2 * BM - 1) / (2 * BM);
    auto waves = [&](int64_t tn) { return (m_tiles * ((a.N + tn - 1) / tn) + pairs - 1) / pairs; };
    return waves(384) * 384 * 96 < waves(256) * 256 * 100;
}

cudaError_t launch_scaled_gemm(const GemmArgs& args, int num_sms, cudaStream_t stream) {
    if (args.G > MAX_GROUPS) return cudaErrorInvalidValue;
    const bool col_alpha = args.G == 0 && args.alpha_b_scope == 2;   // per-output-column factor (dense only)
    // 256-column tiles with one accumulator, dense and grouped alike: for the grouped MoE shapes (K = 2048
    // and 768) they measured faster than 128-column tiles with two accumulators (whose epilogue overlaps
    // the next tile's MMAs but which read A twice as often): gate_up 0.118 against 0.146 ms, down 0.110
    // against 0.132 ms (NVFP4; MXFP8 likewise)
    if (args.fmt == 0) {
        if (args.G > 0) return launch_pair_impl<0, true, false, 256>(args, num_sms, stream);
        if (!col_alpha && wide_mxfp8_tiles(args, num_sms)) return launch_pair_impl<0, false, false, 384>(args, num_sms, stream);
        return col_alpha ? launch_pair_impl<0, false, true, 256>(args, num_sms, stream)
                         : launch_pair_impl<0, false, false, 256>(args, num_sms, stream);
    }
    // NVFP4 with at most three K stages per tile: the output write dominates, and 64-column staged stores
    // (whole 128-byte lines) beat 16-column ones (K = 768 grouped down 108.6 -> 93.4 us; K = 256 / 768
    // dense 72.5 / 78.0 -> 55.7 / 66.6 us for 65536 x 2048 outputs).  With longer K their single staging
    // buffer per warp makes the drain the slower side (K = 2048 grouped 115 -> 122 us), so those keep
    // the 16-column double-buffered stores
    const bool short_k = args.K / 2 / BKB <= 3;
    if (args.G > 0) {
        if (short_k && args.G <= PairCfg<1, true, 256, 3>::MAX_G) return launch_pair_impl<1, true, false, 256, 3>(args, num_sms, stream);
        return launch_pair_impl<1, true, false, 256>(args, num_sms, stream);
    }
    if (short_k && !col_alpha) return launch_pair_impl<1, false, false, 256, 3>(args, num_sms, stream);
    return col_alpha ? launch_pair_impl<1, false, true, 256>(args, num_sms, stream)
                     : launch_pair_impl<1, false, false, 256>(args, num_sms, stream);
}

cudaError_t launch_dq_gemm(const DqGemmArgs& args, int num_sms, cudaStream_t stream) {
    return args.wgrad ? launch_dq_impl<true>(args, num_sms, stream) : launch_dq_impl<false>(args, num_sms, stream);
}

cudaError_t launch_fp8_blockwise_gemm(const BwGemmArgs& args, int num_sms, cudaStream_t stream) {
    return args.b_row_scales ? launch_bw_impl<128, true>(args, num_sms, stream)
                             : launch_bw_impl<128, false>(args, num_sms, stream);
}

uint32_t read_and_clear_device_status() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_mx_device_status, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    cudaMemcpyToSymbol(g_mx_device_status, &zero, sizeof(zero));
    return v;
}

uint32_t read_and_clear_device_status_on(cudaStream_t stream) {
    unsigned int v = 0;
    static const unsigned int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_mx_device_status, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_mx_device_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return 0xFFFFFFFFu;
    return v;
}

cudaError_t launch_watchdog_selftest(unsigned long long limit_ns, cudaStream_t stream) {
    watchdog_selftest_kernel<<<2, NUM_THREADS, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

}  // namespace mxk
