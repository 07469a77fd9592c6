// bf16 x bf16 (or fp16 x fp16) -> fp32 product C = A.B on the sm_103a tensor
// cores (tcgen05, kind::f16; the template argument picks the operand format).
//
// The same three tiling levels as the SIMT kernel, mapped onto Blackwell's
// asynchronous units ("寄存器Tiling跨架构解析", sections 2.1 and 6: on tensor
// cores the per-thread register tile becomes the matrix instruction's
// accumulator fragment):
//
//  * global tiling — a persistent CTA per SM walks 128 x BN C tiles in
//    grouped order (GROUP_M tile-rows at a time) for L2 reuse; BN is 256, or
//    128 / 64 for short, wide products (M <= 128), where 256-wide tiles
//    would leave most SMs idle (N / 256 tiles);
//  * shared tiling — one TMA producer warp streams 64-deep K-slices of A
//    (128 x 64, K-major) and B (64 x BN, N-major) into a ring of
//    128-byte-swizzled shared-memory buffers (4, 6 or 8 stages, about 192 KB),
//    zero-filled past M, N, K;
//  * accumulator tiling — one thread issues tcgen05.mma (M=128, N=BN, K=16,
//    four per K-slice) into a 128 x BN fp32 accumulator in tensor memory
//    (TMEM), double-buffered (2 x BN columns) so the epilogue of one tile
//    overlaps the MMAs of the next;
//  * epilogue — four warps read the accumulator with tcgen05.ld (one TMEM
//    lane = one row of C per thread) and store fp32 rows with masks.
//
// Barriers: full[s]/empty[s] hand stage s between TMA and MMA; tfull[a]/
// tempty[a] hand accumulator a between MMA and epilogue. Every wait is
// bounded by a time limit; a warp that gives up records a timeout in the
// device error word and raises an abort flag so the other warps stop too.
// Before the CTA exits it waits for its own TMA copies and MMAs in flight and
// frees its tensor memory.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace rtm {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;                 // 64 16-bit values = 128 bytes = one swizzle row
constexpr int UMMA_K = 16;
constexpr int kThreads = 192;          // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kGroupM = 16;
constexpr uint32_t A_STAGE_BYTES = BM * BK * 2;            // 16 KB
constexpr uint32_t B_ATOM_BYTES = BK * 64 * 2;             // 8 KB: 64 k-rows x 64 n

// Sizes that follow from the tile width BN (256, 128 or 64).
template <int BN>
struct Tile {
    static constexpr uint32_t B_STAGE_BYTES = BK * BN * 2;  // 32, 16 or 8 KB
    static constexpr uint32_t STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    static constexpr int STAGES = BN == 256 ? 4 : BN == 128 ? 6 : 8;
    static constexpr uint32_t TMEM_COLS = 2 * BN;           // two accumulators
    static constexpr size_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
};

// Instruction descriptor, kind::f16: D fp32, A and B both bf16 (format 1) or
// both fp16 (format 0), A K-major, B MN-major, N = BN, M = 128.
template <bool F16, int BN>
__host__ __device__ constexpr uint32_t idesc()
{
    return (1u << 4)                               // D format: f32
           | ((F16 ? 0u : 1u) << 7)                // A format
           | ((F16 ? 0u : 1u) << 10)               // B format
           | (0u << 15)                            // A major: K
           | (1u << 16)                            // B major: MN
           | ((uint32_t)(BN >> 3) << 17)           // N / 8
           | ((uint32_t)(BM >> 4) << 24);          // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2),
// descriptor version 1. Offsets in bytes.
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
};

template <int BN>
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int &m0, int &n0)
{
    const int group_size = kGroupM * tiles_n;
    const int group = t / group_size;
    const int first_m = group * kGroupM;
    const int rows = min(tiles_m - first_m, kGroupM);
    const int in_group = t - group * group_size;
    m0 = (first_m + in_group % rows) * BM;
    n0 = (in_group / rows) * BN;
}

__device__ __forceinline__ void give_up(int *err, volatile int *abort)
{
    atomicCAS(err, 0, kDevErrTimeout);
    *abort = 1;
}

template <bool F16, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const Params p)
{
    constexpr int STAGES = Tile<BN>::STAGES;
    constexpr uint32_t STAGE_BYTES = Tile<BN>::STAGE_BYTES;
    constexpr uint32_t TMEM_COLS = Tile<BN>::TMEM_COLS;
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

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);  // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int tiles_m = (p.M + BM - 1) / BM;
    const int tiles_n = (p.N + BN - 1) / BN;
    const int ntiles = tiles_m * tiles_n;
    const int kblocks = (p.K + BK - 1) / BK;
    const uint64_t limit = p.limit_ns;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && !p.mute_producer) {
            uint32_t stage = 0, phase = 0;
            uint32_t issued = 0, issued_parity = 0;  // per-stage bit masks
            for (int t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
                int m0, n0;
                tile_coords<BN>(t, tiles_m, tiles_n, m0, n0);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1, limit, abort)) {
                        give_up(p.err, abort);
                        break;
                    }
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    tma_load_2d(sa, &tmA, &full[stage], kb * BK, m0);
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(sb + j * B_ATOM_BYTES, &tmB, &full[stage], n0 + j * 64,
                                    kb * BK);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // No copy into this CTA's shared memory may outlive it: wait for the
            // last load issued into each stage (immediate on the normal path).
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
            uint32_t acc = 0, acc_phase = 0;
            bool issued_any = false;
            for (int t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, limit, abort)) {
                    give_up(p.err, abort);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                bool ok = true;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, limit, abort)) {
                        give_up(p.err, abort);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_STAGE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        // A: K-major rows of 128 B, 8-row groups 1024 B apart;
                        //    the k-step moves 32 B along the swizzled row.
                        // B: N-major, 64-wide atoms B_ATOM_BYTES apart (LBO),
                        //    8 k-rows per 1024 B group (SBO); the k-step is 16 rows.
                        const uint64_t adesc = sdesc_sw128(sa + kk * UMMA_K * 2, 16, 1024);
                        const uint64_t bdesc =
                            sdesc_sw128(sb + kk * UMMA_K * 128, B_ATOM_BYTES, 1024);
                        umma_f16(d_tmem, adesc, bdesc, idesc<F16, BN>(), (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued_any = true;
                    umma_commit(&empty[stage]);  // frees the stage when these MMAs finish
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok)
                    break;
                umma_commit(&tfull[acc]);  // accumulator ready for the epilogue
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            // Every MMA this thread issued completes before tensor memory is freed.
            if (issued_any) {
                umma_commit(drain);
                volatile int no_abort = 0;
                mbar_wait_bounded(drain, 0, limit, &no_abort);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int quarter = warp & 3;  // this warp may touch TMEM lanes 32*quarter ..
        uint32_t acc = 0, acc_phase = 0;
        for (int t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
            int m0, n0;
            tile_coords<BN>(t, tiles_m, tiles_n, m0, n0);
            if (!mbar_wait_bounded(&tfull[acc], acc_phase, limit, abort)) {
                give_up(p.err, abort);
                break;
            }
            tc_fence_after();
            const int row = m0 + quarter * 32 + lane;
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
            float *crow = p.C + (size_t)row * p.N;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + c * 32, r);
                tmem_wait_ld();
                if (c == BN / 32 - 1) {
                    // Accumulator fully read: hand it back to the MMA warp.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&tempty[acc]);
                }
                if (row < p.M) {
                    const int col = n0 + c * 32;
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        if (col + v * 4 < p.N) {  // N % 8 == 0: all four or none
                            float4 o;
                            o.x = __uint_as_float(r[v * 4 + 0]);
                            o.y = __uint_as_float(r[v * 4 + 1]);
                            o.z = __uint_as_float(r[v * 4 + 2]);
                            o.w = __uint_as_float(r[v * 4 + 3]);
                            *reinterpret_cast<float4 *>(crow + col + v * 4) = o;
                        }
                    }
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Row-major rows x cols 16-bit matrix (bf16 or fp16), box of box_rows x 64
// columns, 128 B swizzle.
static bool encode_map(EncodeTiledFn fn, CUtensorMap *map, const void *base, uint64_t rows,
                       uint64_t cols, uint32_t box_rows, bool f16)
{
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN>
cudaError_t launch_bn(const TcLaunch &L, cudaStream_t stream)
{
    auto fn = reinterpret_cast<EncodeTiledFn>(L.encode_tiled);
    if (!fn)
        return cudaErrorInvalidValue;
    CUtensorMap ta, tb;
    // A: M rows x K cols, boxes of 128 rows (m) x 64 k.
    // B: K rows x N cols, boxes of 64 rows (k) x 64 n.
    if (!encode_map(fn, &ta, L.A, (uint64_t)L.M, (uint64_t)L.K, BM, L.f16 != 0) ||
        !encode_map(fn, &tb, L.B, (uint64_t)L.K, (uint64_t)L.N, BK, L.f16 != 0))
        return cudaErrorInvalidValue;

    auto kernel = L.f16 ? gemm_tc_kernel<true, BN> : gemm_tc_kernel<false, BN>;
    static std::atomic<uint64_t> done[2] = {{0}, {0}};
    const size_t smem_bytes = Tile<BN>::SMEM_BYTES;
    const cudaError_t e = set_smem_limit_once(kernel, (int)smem_bytes, done[L.f16 != 0]);
    if (e != cudaSuccess)
        return e;
    const long long ntiles = (long long)((L.M + BM - 1) / BM) * ((L.N + BN - 1) / BN);
    const int grid = (int)(ntiles < L.sm_count ? ntiles : L.sm_count);
    Params p{L.M, L.N, L.K, L.C, L.err, (unsigned long long)L.wait_limit_ns, L.mute_producer};
    kernel<<<grid, kThreads, smem_bytes, stream>>>(ta, tb, p);
    return cudaGetLastError();
}

} // namespace tc

cudaError_t launch_gemm_bf16_tc_bn(const TcLaunch &L, int bn, cudaStream_t stream)
{
    switch (bn) {
    case 256:
        return tc::launch_bn<256>(L, stream);
    case 128:
        return tc::launch_bn<128>(L, stream);
    case 64:
        return tc::launch_bn<64>(L, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

} // namespace rtm
