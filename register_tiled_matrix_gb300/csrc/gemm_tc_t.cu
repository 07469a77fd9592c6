// bf16 x bf16 (or fp16 x fp16) -> fp32 product C = A.B for short, wide
// products (few rows of A, many columns of B) on the sm_103a tensor cores,
// computed as its transpose C^T = B^T.A^T.
//
// With M <= 128 the product reads B (K x N) once and hardly reuses it: it is
// bound by how fast B streams from HBM. The tensor-core kernels that put M on
// the MMA's 128-row side spend most of every shared-memory stage on a
// 128-row A box that is mostly zero fill, and give at most N / 64 CTAs. Here
// the roles swap ("寄存器Tiling跨架构解析", section 6: the accumulator tile is
// whatever the matrix instruction computes; which operand feeds which side is
// free):
//
//  * global tiling — a CTA owns 128 columns of C (n0 .. n0+127) and MN rows
//    (MN = 32, 64 or 128, the next size >= M) and, when that leaves SMs idle,
//    one of S K-ranges (S = 2, 4 or 8 CTAs of one cluster split K);
//  * shared tiling — one TMA producer thread streams 64-deep K-slices of B
//    (two 64 n x 64 k boxes, the MMA's A operand, MN-major) and of A (one
//    64 k x MN box, the MMA's B operand, K-major) into a 6- to 10-stage ring;
//    nearly every staged byte is B, so up to ~190 KB of B is in flight per SM;
//  * accumulator tiling — tcgen05.mma (M = 128 columns of C, N = MN rows of
//    C, K = 16) into an MN-column fp32 accumulator in tensor memory: TMEM lane
//    i holds column n0 + i of C;
//  * epilogue — with S = 1, four warps read the accumulator (one TMEM lane
//    per thread) and store it: for each row of C the 32 lanes of a warp write
//    32 consecutive floats. With S > 1 each CTA writes its partial 128 x MN
//    tile into its (now idle) stage memory; after a cluster barrier CTA r of
//    the cluster sums columns [r MN / S, (r+1) MN / S) over the S partials,
//    read through distributed shared memory in rank order 0, 1, .., S-1 (so
//    the sum is the same on every run), and stores them; a second cluster
//    barrier keeps every partial alive until all have been read.
//
// The same kernel without the swap (SWAP = false) serves tall, narrow
// products (many rows of A, N <= 128; wider ones up to 256 columns ran faster
// on the CTA-pair kernel): A fills the MMA's 128-row side (K-major), B the N
// side (MN = 64 or 128 columns, MN-major; 256 columns as two tiles measured
// the same as one 256-wide tile with half the stages), TMEM lane i is row
// m0 + i of C, and K is split over a cluster the same way.
//
// Every mbarrier wait is bounded in time; a warp that gives up records
// GEMM_ERR_TIMEOUT in the device error word and every thread still reaches
// both cluster barriers.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace rtm {
namespace tct {

constexpr int BNT = 128;  // the MMA's M: columns of C per CTA (SWAP) or rows (no swap)
constexpr int BK = 64;    // 64 16-bit values = one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t B_ATOM_BYTES = 64 * BK * 2;     // 8 KB: 64 k-rows x 64 n
constexpr uint32_t BT_BYTES = BNT * BK * 2;        // 16 KB per stage on the MMA's 128-row side

template <int MN>
struct Cfg {
    static constexpr uint32_t AT_BYTES = MN * BK * 2;  // 4, 8 or 16 KB per stage on the N side
    static constexpr uint32_t STAGE_BYTES = BT_BYTES + AT_BYTES;
    static constexpr int STAGES = (200 * 1024) / STAGE_BYTES;  // 10, 8 or 6
    static constexpr int PITCH = MN + 4;  // floats per row of a partial tile in shared memory
    static constexpr uint32_t PART_BYTES = BNT * PITCH * 4;
    static constexpr uint32_t TMEM_COLS = MN;
    static constexpr size_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
    static_assert(PART_BYTES <= STAGES * STAGE_BYTES, "partial tile must fit the stage ring");
};

// kind::f16: D fp32, A and B both bf16 (1) or both fp16 (0), N = MN, M = 128.
// SWAP: the MMA's A (= B^T) MN-major, its B (= A^T) K-major; otherwise A
// K-major and B MN-major.
template <bool F16, int MN, bool SWAP>
__host__ __device__ constexpr uint32_t idesc()
{
    return (1u << 4) | ((F16 ? 0u : 1u) << 7) | ((F16 ? 0u : 1u) << 10) |
           ((SWAP ? 1u : 0u) << 15) | ((SWAP ? 0u : 1u) << 16) | ((uint32_t)(MN >> 3) << 17) |
           ((uint32_t)(BNT >> 4) << 24);
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
    int splits;         // CTAs per cluster, each summing one K-range
    int mute_producer;  // failure-detection self-test: issue no loads
    int c_vec;          // C rows 16-byte aligned (float4 row stores without the swap)
};

__device__ __forceinline__ void give_up(int *err, volatile int *abort)
{
    atomicCAS(err, 0, kDevErrTimeout);
    *abort = 1;
}

template <bool F16, int MN, bool SWAP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tct_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const Params p)
{
    using Cf = Cfg<MN>;
    constexpr int STAGES = Cf::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * Cf::STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *done = empty + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.splits;
    const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
    const int unit = blockIdx.x / S;
    int m0, n0;
    if constexpr (SWAP) {
        const int tiles_n = (p.N + BNT - 1) / BNT;
        n0 = (unit % tiles_n) * BNT;
        m0 = (unit / tiles_n) * MN;
    } else {
        const int tiles_m = (p.M + BNT - 1) / BNT;
        m0 = (unit % tiles_m) * BNT;
        n0 = (unit / tiles_m) * MN;
    }
    const int kblocks = (p.K + BK - 1) / BK;
    const int per = (kblocks + S - 1) / S;
    const int kb_begin = min(kblocks, (int)rank * per);
    const int kb_end = min(kblocks, kb_begin + per);
    const uint64_t limit = p.limit_ns;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *abort = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cf::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && !p.mute_producer) {
            uint32_t stage = 0, phase = 0;
            uint32_t issued = 0, issued_parity = 0;
            for (int kb = kb_begin; kb < kb_end && !*abort; ++kb) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1, limit, abort)) {
                    give_up(p.err, abort);
                    break;
                }
                const uint32_t sbig = smem_u32(smem + stage * Cf::STAGE_BYTES);
                const uint32_t ssmall = sbig + BT_BYTES;
                mbar_arrive_expect_tx(&full[stage], Cf::STAGE_BYTES);
                if constexpr (SWAP) {
                    tma_load_2d(sbig, &tmB, &full[stage], n0, kb * BK);
                    tma_load_2d(sbig + B_ATOM_BYTES, &tmB, &full[stage], n0 + 64, kb * BK);
                    tma_load_2d(ssmall, &tmA, &full[stage], kb * BK, m0);
                } else {
                    tma_load_2d(sbig, &tmA, &full[stage], kb * BK, m0);
#pragma unroll
                    for (int j = 0; j < MN / 64; ++j)
                        tma_load_2d(ssmall + j * B_ATOM_BYTES, &tmB, &full[stage], n0 + 64 * j,
                                    kb * BK);
                }
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            // No copy into this CTA's shared memory may outlive it.
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s)) {
                    volatile int no_abort = 0;
                    mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, limit, &no_abort);
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool issued_any = false;
            for (int kb = kb_begin; kb < kb_end; ++kb) {
                if (!mbar_wait_bounded(&full[stage], phase, limit, abort)) {
                    give_up(p.err, abort);
                    break;
                }
                tc_fence_after();
                const uint32_t sbig = smem_u32(smem + stage * Cf::STAGE_BYTES);
                const uint32_t ssmall = sbig + BT_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                    // MN-major side: 64-wide atoms B_ATOM_BYTES apart, 16 k-rows per step.
                    // K-major side: rows of 128 B, 8-row groups 1024 B apart, 32 B per step.
                    uint64_t adesc, bdesc;
                    if constexpr (SWAP) {
                        adesc = sdesc_sw128(sbig + kk * UMMA_K * 128, B_ATOM_BYTES, 1024);
                        bdesc = sdesc_sw128(ssmall + kk * UMMA_K * 2, 16, 1024);
                    } else {
                        adesc = sdesc_sw128(sbig + kk * UMMA_K * 2, 16, 1024);
                        bdesc = sdesc_sw128(ssmall + kk * UMMA_K * 128, B_ATOM_BYTES, 1024);
                    }
                    umma_f16(tmem_base, adesc, bdesc, idesc<F16, MN, SWAP>(),
                             (kb != kb_begin || kk != 0) ? 1u : 0u);
                }
                issued_any = true;
                umma_commit(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (issued_any) {
                umma_commit(done);
                volatile int no_abort = 0;
                mbar_wait_bounded(done, 0, limit, &no_abort);  // before TMEM is freed
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // TMEM lane: column n0 + row (SWAP) or row m0 + row of C
        const bool have = kb_end > kb_begin;
        bool ok = true;
        if (have && !mbar_wait_bounded(done, 0, limit, abort)) {
            give_up(p.err, abort);
            ok = false;
        }
        tc_fence_after();
        const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16);
        if (S == 1) {
            if (ok) {
#pragma unroll 1
                for (int c = 0; c < MN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + c * 32, r);
                    tmem_wait_ld();
                    if constexpr (SWAP) {
                        const int gn = n0 + row;
                        const int rows = min(32, p.M - (m0 + c * 32));
                        if (gn < p.N) {
                            float *cp = p.C + (size_t)(m0 + c * 32) * p.N + gn;
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j < rows)
                                    cp[(size_t)j * p.N] = __uint_as_float(r[j]);
                        }
                    } else {
                        const int gm = m0 + row;
                        const int col = n0 + c * 32;
                        if (gm < p.M) {
                            float *cp = p.C + (size_t)gm * p.N + col;
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                if (p.c_vec && col + 4 * v + 3 < p.N) {
                                    *reinterpret_cast<float4 *>(cp + 4 * v) = make_float4(
                                        __uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                        __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                                } else {
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        if (col + 4 * v + e < p.N)
                                            cp[4 * v + e] = __uint_as_float(r[4 * v + e]);
                                }
                            }
                        }
                    }
                }
            }
        } else {
            float *part = reinterpret_cast<float *>(smem);
#pragma unroll 1
            for (int c = 0; c < MN / 32; ++c) {
                uint32_t r[32];
                if (have && ok) {
                    tmem_ld_32x32b_x32(t_row + c * 32, r);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        r[j] = 0u;  // an empty K-range contributes zeros
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<uint4 *>(part + row * Cf::PITCH + c * 32 + 4 * q) =
                        make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
            }
        }
    }

    if (S > 1) {
        cluster_sync();  // every partial tile of the cluster is in shared memory
        if (warp >= 2) {
            const int row = (warp & 3) * 32 + lane;
            const int cols = MN / S;
            const int c0 = (int)rank * cols;
            const uint32_t mine = smem_u32(smem) + (uint32_t)(row * Cf::PITCH) * 4u;
            for (int cc = 0; cc < cols; cc += 4) {
                const uint32_t off = (uint32_t)(c0 + cc) * 4u;
                float4 acc = ld_shared_cluster_v4(mapa_shared(mine + off, 0));
                for (int q = 1; q < S; ++q) {
                    const float4 v = ld_shared_cluster_v4(mapa_shared(mine + off, (uint32_t)q));
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
                if constexpr (SWAP) {
                    const int gn = n0 + row;
                    const int gm = m0 + c0 + cc;
                    if (gn < p.N) {
                        float *cp = p.C + (size_t)gm * p.N + gn;
                        if (gm + 0 < p.M) cp[0] = acc.x;
                        if (gm + 1 < p.M) cp[(size_t)p.N] = acc.y;
                        if (gm + 2 < p.M) cp[(size_t)2 * p.N] = acc.z;
                        if (gm + 3 < p.M) cp[(size_t)3 * p.N] = acc.w;
                    }
                } else {
                    const int gm = m0 + row;
                    const int gn = n0 + c0 + cc;
                    if (gm < p.M) {
                        float *cp = p.C + (size_t)gm * p.N + gn;
                        if (p.c_vec && gn + 3 < p.N) {
                            *reinterpret_cast<float4 *>(cp) = acc;
                        } else {
                            if (gn + 0 < p.N) cp[0] = acc.x;
                            if (gn + 1 < p.N) cp[1] = acc.y;
                            if (gn + 2 < p.N) cp[2] = acc.z;
                            if (gn + 3 < p.N) cp[3] = acc.w;
                        }
                    }
                }
            }
        }
        cluster_sync();  // no CTA leaves while a peer may still read its partial
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cf::TMEM_COLS);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static bool encode_map(EncodeTiledFn fn, CUtensorMap *map, const void *base, uint64_t rows,
                       uint64_t cols, uint32_t box_rows, bool f16)
{
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <bool F16, int MN, bool SWAP>
static cudaError_t launch_mn(const TcLaunch &L, int splits, cudaStream_t stream)
{
    using Cf = Cfg<MN>;
    auto fn = reinterpret_cast<EncodeTiledFn>(L.encode_tiled);
    if (!fn)
        return cudaErrorInvalidValue;
    CUtensorMap ta, tb;
    // A: M x K, boxes of 64 k x (MN rows with the swap, 128 without);
    // B: K x N, boxes of 64 k-rows x 64 n.
    if (!encode_map(fn, &ta, L.A, (uint64_t)L.M, (uint64_t)L.K, SWAP ? MN : BNT, F16) ||
        !encode_map(fn, &tb, L.B, (uint64_t)L.K, (uint64_t)L.N, BK, F16))
        return cudaErrorInvalidValue;
    auto kernel = gemm_tct_kernel<F16, MN, SWAP>;
    static std::atomic<uint64_t> done{0};
    cudaError_t e = set_smem_limit_once(kernel, (int)Cf::SMEM_BYTES, done);
    if (e != cudaSuccess)
        return e;
    const long long tiles = SWAP ? (long long)((L.N + BNT - 1) / BNT) * ((L.M + MN - 1) / MN)
                                 : (long long)((L.M + BNT - 1) / BNT) * ((L.N + MN - 1) / MN);
    // Every cluster resident at once (CTAs wait for their cluster's partials):
    // halve the split while more clusters would be launched than fit.
    static std::atomic<int> resident[4][64] = {};  // clusters of 1, 2, 4, 8
    while (splits > 1) {
        const int slot = splits == 2 ? 1 : splits == 4 ? 2 : 3;
        const int fit = resident_clusters(kernel, splits, kThreads, Cf::SMEM_BYTES, resident[slot]);
        if (fit <= 0 || tiles <= fit)
            break;
        splits /= 2;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * splits), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cf::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int c_vec = (L.N % 4 == 0) && ((reinterpret_cast<uintptr_t>(L.C) & 15) == 0);
    Params p{L.M, L.N, L.K, L.C, L.err, (unsigned long long)L.wait_limit_ns, splits,
             L.mute_producer, c_vec};
    return cudaLaunchKernelEx(&cfg, kernel, ta, tb, p);
}

} // namespace tct

int tct_rows(int M)
{
    return M <= 32 ? 32 : M <= 64 ? 64 : 128;
}

int tcs_cols(int N)
{
    return N <= 64 ? 64 : 128;
}

cudaError_t launch_gemm_tc_t(const TcLaunch &L, int splits, bool swap, cudaStream_t stream)
{
    using namespace tct;
    if (splits != 1 && splits != 2 && splits != 4 && splits != 8)
        return cudaErrorInvalidValue;
    if (swap) {
        const int mn = tct_rows(L.M);
        if (L.f16)
            return mn == 32 ? launch_mn<true, 32, true>(L, splits, stream)
                   : mn == 64 ? launch_mn<true, 64, true>(L, splits, stream)
                              : launch_mn<true, 128, true>(L, splits, stream);
        return mn == 32 ? launch_mn<false, 32, true>(L, splits, stream)
               : mn == 64 ? launch_mn<false, 64, true>(L, splits, stream)
                          : launch_mn<false, 128, true>(L, splits, stream);
    }
    const int mn = tcs_cols(L.N);
    if (L.f16)
        return mn == 64 ? launch_mn<true, 64, false>(L, splits, stream)
                        : launch_mn<true, 128, false>(L, splits, stream);
    return mn == 64 ? launch_mn<false, 64, false>(L, splits, stream)
                    : launch_mn<false, 128, false>(L, splits, stream);
}

} // namespace rtm
