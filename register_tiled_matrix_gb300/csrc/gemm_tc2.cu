// bf16 x bf16 (or fp16 x fp16) -> fp32 product C = A.B on CTA pairs: the
// two-SM form of tcgen05 (cta_group::2) on sm_103a.
//
// Same tiling levels as gemm_tc.cu ("寄存器Tiling跨架构解析", sections 2.1 and
// 6: on tensor cores the register tile becomes the matrix instruction's
// accumulator), with one change that matters on Blackwell: a cluster of two
// CTAs on the two SMs of a pair computes a 256 x 256 C tile with one MMA
// instruction stream. Each CTA stages only its own half of the operands —
// 128 rows of A and 128 columns of B per 64-deep K-slice, 32 KB instead of
// the 48 KB a lone 128 x 256 tile needs — so the bytes every SM must pull
// from L2 per tensor-core cycle fall by a third, while each SM still keeps a
// 128 x 256 fp32 accumulator in its own tensor memory.
//
//  * global tiling — persistent clusters walk 256 x 256 tiles in groups of
//    GROUP_M tile-rows (L2 reuse);
//  * shared tiling — in each CTA one thread issues the TMA boxes of its
//    halves into a 6-stage ring; the copies of both CTAs signal one mbarrier
//    in the even CTA, which expects the pair's 64 KB per stage;
//  * accumulator tiling — one thread of the even CTA issues
//    tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): rows 0-127 land in
//    the even CTA's tensor memory, rows 128-255 in the odd CTA's; completions
//    are multicast to the stage and accumulator barriers of both CTAs;
//    accumulators are double-buffered (2 x 256 columns);
//  * epilogue — in each CTA four warps read their CTA's accumulator rows
//    with tcgen05.ld and store them; the eight epilogue warps of the pair hand
//    the accumulator back to the even CTA. Where C rows are 16-byte aligned
//    (N % 4 == 0, C 16-byte aligned) each warp stages its 32 x 32 blocks in
//    128-byte-swizzled shared memory and the TMA unit stores them (a float4
//    per lane and row before: 0.605 ms at 8192^3, 0.111 ms at 8192^2 x 64;
//    TMA stores: 0.582 and 0.054); otherwise each warp turns its 32 x 32 block
//    around in shared memory and stores it row by row, 32 consecutive floats
//    per store instruction.
//
// The operands' row strides are parameters of the tensor maps, so the kernel
// also runs on copies of A or B whose rows were padded to 16-byte multiples.
//
// Products whose tiles would occupy at most half the pairs (256 x 8192 x 8192:
// 32 tiles for 76 pairs) split K in two: the persistent loop walks (tile, K
// half) units, C is zero-filled first, and the epilogue adds each half's tile
// into C with TMA reduce-adds. With exactly two partials the sum 0 + a + b is
// the same in either order (IEEE addition is commutative), so results still
// repeat exactly from call to call.
//
// Every mbarrier wait is bounded in time (see gemm_tc.cu); the cluster
// barriers at start and end are reached on every path.
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace rtm {
namespace tc2 {

constexpr int PM = 256;            // pair tile rows (128 per CTA)
constexpr int PN = 256;            // pair tile columns
constexpr int HM = 128;            // A rows staged per CTA
constexpr int HN = 128;            // B columns staged per CTA
constexpr int BK = 64;             // 64 16-bit values = one 128-byte swizzle row
constexpr int STAGES = 6;
constexpr int UMMA_K = 16;
constexpr int kThreads = 192;      // warp 0 TMA, warp 1 MMA (even CTA), warps 2-5 epilogue
constexpr int kGroupM = 8;
constexpr uint32_t A_BYTES = HM * BK * 2;          // 16 KB
constexpr uint32_t B_ATOM_BYTES = BK * 64 * 2;     // 8 KB: 64 k-rows x 64 columns
constexpr uint32_t B_BYTES = BK * HN * 2;          // 16 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t PAIR_STAGE_BYTES = 2 * STAGE_BYTES;
constexpr uint32_t TMEM_COLS = 2 * PN;             // 512: two accumulators
constexpr size_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr int kEpiPitch = 33;                      // floats per row of an epilogue block
constexpr uint32_t EPI_WARP_BYTES = 32 * kEpiPitch * 4;
constexpr size_t SMEM_BYTES_SCALAR_C = SMEM_BYTES + 4 * EPI_WARP_BYTES;
// TMA-store epilogue: per epilogue warp two 32 x 32 fp32 boxes (4 KB each,
// 128-byte swizzled, 1024-byte aligned) after a 1 KB block for the barriers.
constexpr uint32_t EPI_BOX_BYTES = 32 * 32 * 4;
constexpr size_t SMEM_BYTES_TMA_C = SMEM_BYTES + 1024 + 4 * 2 * EPI_BOX_BYTES;
// Epilogue variants: C rows 16-byte aligned (N % 4 == 0, C 16-byte aligned),
// TMA stores of 32 x 32 boxes; any other C, row-by-row stores through shared
// memory.
enum { kEpiRowByRow = 1, kEpiTmaStore = 2 };
constexpr uint16_t kBothCtas = 0x3;
constexpr uint16_t kEvenCta = 0x1;

// kind::f16 instruction descriptor for the pair: D fp32, A/B bf16 (1) or fp16
// (0), A K-major, B MN-major, N = 256, M = 256.
template <bool F16>
__host__ __device__ constexpr uint32_t idesc()
{
    return (1u << 4) | ((F16 ? 0u : 1u) << 7) | ((F16 ? 0u : 1u) << 10) | (0u << 15) |
           (1u << 16) | ((uint32_t)(PN >> 3) << 17) | ((uint32_t)(PM >> 4) << 24);
}

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

struct Params {
    int M, N, K;
    float *C;
    int *err;
    unsigned long long limit_ns;
    int mute_producer;
    int split_from;  // tiles from here on: K halves added into a zeroed C (TMA-store
                     // epilogue only); the tile count for none
};

// Work unit u of the persistent loop: tiles before split_from are one unit
// each (all K-blocks), every later tile two units, its K halves (each half
// non-empty: the host splits only K of at least two blocks). A split unit adds
// its tile into C instead of storing it.
__device__ __forceinline__ void unit_of(int u, int split_from, int kblocks, int &tile,
                                        int &kb_begin, int &kb_end, bool &split)
{
    if (u < split_from) {
        tile = u;
        kb_begin = 0;
        kb_end = kblocks;
        split = false;
    } else {
        const int v = u - split_from;
        const int per = (kblocks + 1) / 2;
        tile = split_from + (v >> 1);
        kb_begin = (v & 1) * per;
        kb_end = min(kblocks, kb_begin + per);
        split = true;
    }
}

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int &m0, int &n0)
{
    const int group_size = kGroupM * tiles_n;
    const int group = t / group_size;
    const int first_m = group * kGroupM;
    const int rows = min(tiles_m - first_m, kGroupM);
    const int in_group = t - group * group_size;
    m0 = (first_m + in_group % rows) * PM;
    n0 = (in_group / rows) * PN;
}

__device__ __forceinline__ void give_up(int *err, volatile int *abort)
{
    atomicCAS(err, 0, kDevErrTimeout);
    *abort = 1;
}

template <bool F16, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: the even CTA, which issues the MMAs
    const bool even = rank == 0;
    const int cluster_id = blockIdx.x >> 1;
    const int num_clusters = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);   // even CTA: its producer's expect_tx arrival
            mbar_init(&empty[s], 1);  // one multicast commit per stage use
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);  // even CTA: the pair's eight epilogue warps
        }
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if constexpr (EPI == kEpiTmaStore)
            tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int tiles_m = (p.M + PM - 1) / PM;
    const int tiles_n = (p.N + PN - 1) / PN;
    const int split_from = p.split_from;
    const int nunits = split_from + 2 * (tiles_m * tiles_n - split_from);
    const int kblocks = (p.K + BK - 1) / BK;
    const uint64_t limit = p.limit_ns;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0 && !p.mute_producer) {
            uint32_t stage = 0, phase = 0;
            uint32_t issued = 0, issued_parity = 0;
            for (int u = cluster_id; u < nunits && !*abort; u += num_clusters) {
                int m0, n0, tile, kb_begin, kb_end;
                bool split;
                unit_of(u, split_from, kblocks, tile, kb_begin, kb_end, split);
                tile_coords(tile, tiles_m, tiles_n, m0, n0);
                const int row0 = m0 + (int)rank * HM;
                const int col0 = n0 + (int)rank * HN;
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1, limit, abort)) {
                        give_up(p.err, abort);
                        break;
                    }
                    if (even)
                        mbar_arrive_expect_tx(&full[stage], PAIR_STAGE_BYTES);
                    const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    tma_load_2d_pair(sa, &tmA, fb, kb * BK, row0);
                    tma_load_2d_pair(sb, &tmB, fb, col0, kb * BK);
                    tma_load_2d_pair(sb + B_ATOM_BYTES, &tmB, fb, col0 + 64, kb * BK);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // No copy into this CTA's shared memory may outlive the pair.
            if (even) {
                for (int s = 0; s < STAGES; ++s)
                    if (issued & (1u << s)) {
                        volatile int no_abort = 0;
                        mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, limit, &no_abort);
                    }
            } else if (issued && *abort) {
                // The odd CTA's copies signal the even CTA's barriers; on the
                // abort path give them time to land before leaving.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA)
        if (even && lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool issued_any = false;
            for (int u = cluster_id; u < nunits && !*abort; u += num_clusters) {
                int tile, kb_begin, kb_end;
                bool split;
                unit_of(u, split_from, kblocks, tile, kb_begin, kb_end, split);
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, limit, abort)) {
                    give_up(p.err, abort);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * PN;
                bool ok = true;
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, limit, abort)) {
                        give_up(p.err, abort);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint64_t adesc = sdesc_sw128(sa + kk * UMMA_K * 2, 16, 1024);
                        const uint64_t bdesc =
                            sdesc_sw128(sb + kk * UMMA_K * 128, B_ATOM_BYTES, 1024);
                        umma_f16_pair(d_tmem, adesc, bdesc, idesc<F16>(),
                                      (kb > kb_begin || kk > 0) ? 1u : 0u);
                    }
                    issued_any = true;
                    umma_commit_pair_multicast(&empty[stage], kBothCtas);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok)
                    break;
                umma_commit_pair_multicast(&tfull[acc], kBothCtas);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            if (issued_any) {
                umma_commit_pair_multicast(drain, kEvenCta);
                volatile int no_abort = 0;
                mbar_wait_bounded(drain, 0, limit, &no_abort);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (both CTAs)
        const int quarter = warp & 3;
        uint32_t acc = 0, acc_phase = 0;
        for (int u = cluster_id; u < nunits && !*abort; u += num_clusters) {
            int m0, n0, tile, kb_begin, kb_end;
            bool split;
            unit_of(u, split_from, kblocks, tile, kb_begin, kb_end, split);
            tile_coords(tile, tiles_m, tiles_n, m0, n0);
            if (!mbar_wait_bounded(&tfull[acc], acc_phase, limit, abort)) {
                give_up(p.err, abort);
                break;
            }
            tc_fence_after();
            if constexpr (EPI == kEpiRowByRow) {
                // Lane i holds row i of a 32 x 32 block: write it to shared memory
                // as row i (pitch 33 floats, so the 32 lanes hit 32 banks), then
                // read it back by columns so lane j stores column j of each row.
                float *blk = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES + 256 +
                                                       quarter * EPI_WARP_BYTES);
                const int row0 = m0 + (int)rank * HM + quarter * 32;
                const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * PN;
#pragma unroll 1
                for (int c = 0; c < PN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + c * 32, r);
                    tmem_wait_ld();
                    if (c == PN / 32 - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive_cluster_tmem_free(mapa_shared(smem_u32(&tempty[acc]), 0));
                    }
#pragma unroll
                    for (int v = 0; v < 32; ++v)
                        blk[lane * kEpiPitch + v] = __uint_as_float(r[v]);
                    __syncwarp();
                    const int col = n0 + c * 32 + lane;
                    const int rows = min(32, p.M - row0);
                    if (col < p.N) {
                        float *cp = p.C + (size_t)row0 * p.N + col;
#pragma unroll 4
                        for (int rr = 0; rr < rows; ++rr)
                            cp[(size_t)rr * p.N] = blk[rr * kEpiPitch + lane];
                    }
                    __syncwarp();
                }
            } else {
                // Lane i writes row i of each 32 x 32 block into a 128-byte-
                // swizzled box (16-byte chunk q of row i at q ^ (i mod 8):
                // 8 lanes cover all 32 banks), then one lane hands the box to
                // the TMA unit, which stores it (or, K split, adds it) and
                // clips rows and columns outside M x N. Two blocks per pass,
                // one per box: both tensor-memory loads share one wait, both
                // boxes one proxy fence and one bulk group (one block per
                // pass took 0.3 us of dependent latency each, 2.4 us a tile).
                // A box is rewritten only after the store issued from it has
                // read it.
                uint8_t *boxes = smem + STAGES * STAGE_BYTES + 1024 + quarter * 2 * EPI_BOX_BYTES;
                const int row0 = m0 + (int)rank * HM + quarter * 32;
                const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * PN;
#pragma unroll 1
                for (int c = 0; c < PN / 32; c += 2) {
                    uint32_t r[2][32];
                    tmem_ld_32x32b_x32(t_row + c * 32, r[0]);
                    tmem_ld_32x32b_x32(t_row + (c + 1) * 32, r[1]);
                    tmem_wait_ld();
                    if (c + 2 == PN / 32) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive_cluster_tmem_free(mapa_shared(smem_u32(&tempty[acc]), 0));
                    }
                    if (row0 >= p.M || n0 + c * 32 >= p.N)
                        continue;  // both boxes lie outside C
                    const bool second = n0 + (c + 1) * 32 < p.N;
                    if (lane == 0)
                        bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int b = 0; b < 2; ++b)
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            *reinterpret_cast<uint4 *>(boxes + b * EPI_BOX_BYTES + lane * 128 +
                                                       ((q ^ (lane & 7)) << 4)) =
                                make_uint4(r[b][4 * q], r[b][4 * q + 1], r[b][4 * q + 2],
                                           r[b][4 * q + 3]);
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        if (split)
                            grid_dependency_wait();  // C zeroed by the preceding fill
                        for (int b = 0; b < (second ? 2 : 1); ++b) {
                            const uint32_t src = smem_u32(boxes + b * EPI_BOX_BYTES);
                            const int col = n0 + (c + b) * 32;
                            if (split)
                                tma_reduce_add_2d(&tmC, src, col, row0);
                            else
                                tma_store_2d(&tmC, src, col, row0);
                        }
                        bulk_commit_group();
                    }
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        if constexpr (EPI == kEpiTmaStore) {
            if (lane == 0)
                bulk_wait_group<0>();  // every store done before the CTA leaves
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still signal or read it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// Zero the C tiles from tile `first` on (those whose K halves are added into
// C), clipped to M x N: one CTA per tile, float4 stores (this path has C rows
// on 16-byte boundaries, N % 4 == 0, so every clipped row is whole float4s).
__global__ void zero_tiles_kernel(float *C, int M, int N, int first)
{
    grid_launch_dependents();  // the pair kernel waits for these zeros only before adding
    int m0, n0;
    tile_coords(first + (int)blockIdx.x, (M + PM - 1) / PM, (N + PN - 1) / PN, m0, n0);
    const int rows = min(PM, M - m0), quads = min(PN, N - n0) / 4;
    for (int i = threadIdx.x; i < rows * quads; i += blockDim.x) {
        const int r = i / quads, q = i - r * quads;
        *reinterpret_cast<float4 *>(C + (size_t)(m0 + r) * N + n0 + 4 * q) =
            make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// rows x cols matrix of 2-byte values whose rows are `ld` values apart
// (ld >= cols, ld * 2 a multiple of 16); columns past `cols` are never read.
static bool encode_map(EncodeTiledFn fn, CUtensorMap *map, const void *base, uint64_t rows,
                       uint64_t cols, uint64_t ld, uint32_t box_rows, bool f16)
{
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// C (M x N fp32, rows N * 4 bytes apart, N % 4 == 0, 16-byte aligned) as
// 32 x 32 boxes with the 128-byte swizzle of the epilogue's staging boxes.
static bool encode_c_map(EncodeTiledFn fn, CUtensorMap *map, const void *base, uint64_t rows,
                         uint64_t cols)
{
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

} // namespace tc2

cudaError_t launch_gemm_tc_pair(const TcLaunch &L, cudaStream_t stream)
{
    return launch_gemm_tc_pair_split(L, 0, stream);
}

cudaError_t launch_gemm_tc_pair_split(const TcLaunch &L, int splits, cudaStream_t stream)
{
    using namespace tc2;
    auto fn = reinterpret_cast<EncodeTiledFn>(L.encode_tiled);
    if (!fn)
        return cudaErrorInvalidValue;
    CUtensorMap ta, tb;
    // A: M x K, boxes of 128 rows x 64 k; B: K x N, boxes of 64 k-rows x 64 n.
    const uint64_t lda = L.lda > 0 ? (uint64_t)L.lda : (uint64_t)L.K;
    const uint64_t ldb = L.ldb > 0 ? (uint64_t)L.ldb : (uint64_t)L.N;
    if (!encode_map(fn, &ta, L.A, (uint64_t)L.M, (uint64_t)L.K, lda, HM, L.f16 != 0) ||
        !encode_map(fn, &tb, L.B, (uint64_t)L.K, (uint64_t)L.N, ldb, BK, L.f16 != 0))
        return cudaErrorInvalidValue;
    const bool c_vec = (L.N % 4 == 0) && ((reinterpret_cast<uintptr_t>(L.C) & 15) == 0);
    CUtensorMap tc;
    std::memset(&tc, 0, sizeof(tc));
    if (c_vec && !encode_c_map(fn, &tc, L.C, (uint64_t)L.M, (uint64_t)L.N))
        return cudaErrorInvalidValue;
    auto kernel = L.f16 ? (c_vec ? gemm_tc2_kernel<true, kEpiTmaStore>
                                 : gemm_tc2_kernel<true, kEpiRowByRow>)
                        : (c_vec ? gemm_tc2_kernel<false, kEpiTmaStore>
                                 : gemm_tc2_kernel<false, kEpiRowByRow>);
    const size_t smem_bytes = c_vec ? SMEM_BYTES_TMA_C : SMEM_BYTES_SCALAR_C;
    const int fi = (L.f16 != 0 ? 1 : 0) + (c_vec ? 0 : 2);
    static std::atomic<uint64_t> done[4] = {{0}, {0}, {0}, {0}};
    cudaError_t e = set_smem_limit_once(kernel, (int)smem_bytes, done[fi]);
    if (e != cudaSuccess)
        return e;
    // How many pairs can be resident at once (the persistent grid), cached
    // per device and kernel; 0 means not yet known.
    static std::atomic<int> max_clusters[4][64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    int clusters_max = (dev >= 0 && dev < 64) ? max_clusters[fi][dev].load() : 0;
    if (clusters_max <= 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (L.sm_count / 2), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem_bytes;
        if (cudaOccupancyMaxActiveClusters(&clusters_max, kernel, &cfg) != cudaSuccess ||
            clusters_max <= 0) {
            cudaGetLastError();
            clusters_max = L.sm_count / 2;
        }
        if (dev >= 0 && dev < 64)
            max_clusters[fi][dev].store(clusters_max);
    }
    const long long ntiles = (long long)((L.M + PM - 1) / PM) * ((L.N + PN - 1) / PN);
    // splits == 0: choose (pair_split_from, tc_plan.cu); 1: no split; 2: every tile.
    const int kblocks = (L.K + BK - 1) / BK;
    if (splits < 0 || splits > 2)
        return cudaErrorInvalidValue;
    const long long split_from = splits == 2   ? 0
                                 : splits == 1 ? ntiles
                                               : pair_split_from(ntiles, clusters_max, kblocks, c_vec);
    if (split_from < ntiles && (!c_vec || kblocks < 2))
        return cudaErrorInvalidValue;
    const long long nunits = split_from + 2 * (ntiles - split_from);
    const int clusters = (int)(nunits < clusters_max ? nunits : clusters_max);
    if (split_from == 0) {
        e = launch_zero_fill(L.C, (int64_t)L.M * L.N, stream);
    } else if (split_from < ntiles) {
        zero_tiles_kernel<<<(unsigned)(ntiles - split_from), 256, 0, stream>>>(L.C, L.M, L.N,
                                                                             (int)split_from);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess)
        return e;
    Params p{L.M, L.N, L.K, L.C, L.err, (unsigned long long)L.wait_limit_ns, L.mute_producer,
             (int)split_from};
    // After a zero fill the kernel is a programmatic dependent of it: its main
    // loop reads only A and B, and each split unit waits for the fill (and its
    // memory) before its first reduce-add, so the fill and its launch overlap
    // the main loop.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = split_from < ntiles ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, ta, tb, tc, p);
}

} // namespace rtm
