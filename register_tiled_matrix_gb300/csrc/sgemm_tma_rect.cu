// SIMT FP32 product C = A.B on rectangular C tiles fed by the tensor-memory-
// access (TMA) unit: 256 x 64 tiles for tall, narrow products (N <= 64) and
// 64 x 256 tiles for short ones (33 <= M <= 64), K split over the CTAs of a
// thread-block cluster or not.
//
// The register level is the cp.async kernel's (sgemm_simt.cu) for the same
// tiles: 16 x 16 threads, (BM / 16) x (BN / 16) accumulators per thread as
// 4 x 4 sub-blocks spaced 64 rows or columns apart, 32-deep K slices, and per
// k BM / 64 LDS.128 of A and BN / 64 of B feeding 64 FMAs, here as 32 packed
// two-wide FMAs ("理解 Register Tiling", section "关键循环"; "寄存器Tiling跨架构解析",
// sections 1.1 and 6.3). As in sgemm_tma.cu, one thread issues two TMA loads
// per slice — a BM m x 32 k box of A (row-major, 128-byte swizzle) into a
// staging tile and a 32 k x BN n box of B into a B stage — and the threads
// transpose A into the k-major layout the fragment loads read (4 x 4 blocks,
// 4 LDS.128 + 4 STS.128 each). In the cp.async kernel every thread issued
// 34 (tall) or 24 (short) copies per slice for the same data.
//
// The 256-row tiles have one k-major A stage: two would need 114 KB of
// shared memory and one CTA per SM; with one the CTA needs 81 KB, two CTAs
// share an SM, and each covers the other's transpose. Per slice: wait for the
// slice's loads, transpose A, a CTA barrier, thread 0 issues the next slice
// (its A into the free staging tile, its B into the other B stage), the k
// loop, a CTA barrier (the A stage is free again). The 64-row tiles have two
// A stages (90 KB) and the pipeline of sgemm_tma.cu: one barrier per slice.
//
// K is split over the S CTAs of a cluster (grid (tiles, S), cluster (1, S, 1),
// S in {1, 2, 4, 8}); each parks its partial tile in its shared memory and,
// after a cluster barrier, adds rows [rank * BM / S, +BM / S) of the S
// partials read through distributed shared memory in rank order (the same
// sum on every call), then stores them; a second barrier keeps the partials
// alive until read. Every mbarrier wait is bounded; a wait that gives up
// records GEMM_ERR_TIMEOUT and raises the CTA's abort flag, after which
// thread 0 issues nothing more, and every thread still reaches every barrier.
//
// Requirements (checked by the launcher): K % 4 == 0, N % 4 == 0, A and B
// 16-byte aligned (TMA row strides and bases).
#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"
#include "simt_tma_common.cuh"

namespace rtm {
namespace simt_tma_rect {

constexpr int kThreads = 256;
constexpr int BK = 32;
constexpr int kGroupM = 16;          // tile-rows per L2 group
constexpr int kSpreadSmem = 120 * 1024;  // more than half of an SM: one CTA per SM

// Shared-memory layout in bytes from a 1024-byte-aligned base: staging tile
// (BM rows of 128 bytes, 128-byte swizzle), two B stages, one k-major A stage
// (rows padded to BM + 4 floats: conflict-free stores and reads), two
// mbarriers; the partial tile of the cluster split (rows padded to BN + 4)
// reuses the stages.
template <int BM, int BN>
struct Shape {
    static_assert((BM == 256 && BN == 64) || (BM == 64 && BN == 256), "tall or short tiles");
    static constexpr int TM = BM / 16, TN = BN / 16;  // accumulators per thread
    static constexpr int LDA = BM + 4;
    static constexpr int A_STAGE = BK * LDA;          // floats
    static constexpr int B_STAGE = BK * BN;           // floats
    // Two A stages where two CTAs still fit on an SM (the 64-row tiles): the
    // transpose of slice s + 1 then overlaps slice s's k loop, one barrier
    // per slice; the 256-row tiles keep one.
    static constexpr int A_STAGES = (BM * BK + 2 * BK * BN + 2 * BK * LDA) * 4 + 2048 <= 113 * 1024 ? 2 : 1;
    static constexpr int OFF_ST = 0;
    static constexpr int OFF_B = BM * BK * 4;
    static constexpr int OFF_A = OFF_B + 2 * B_STAGE * 4;
    static constexpr int OFF_BAR = OFF_A + A_STAGES * A_STAGE * 4;
    static constexpr int SMEM_BYTES = OFF_BAR + 16 + 1024;  // + room to align the base
    static constexpr uint32_t kSliceBytes = (BM * BK + BK * BN) * 4;
    static constexpr int kPartPitch = BN + 4;
    static_assert(BM * kPartPitch * 4 <= OFF_BAR, "the partial tile fits below the barriers");
    static_assert(2 * (SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs per SM");
};

using simt_tma_common::EncodeTiledFn;
using simt_tma_common::encode_f32_map;
using simt_tma_common::lds128;
using simt_tma_common::sts128;

__device__ __forceinline__ void tile_of_block(int bid, int tiles_m, int tiles_n, int &tile_m,
                                              int &tile_n)
{
    simt_tma_common::grouped_tile<kGroupM>(bid, tiles_m, tiles_n, tile_m, tile_n);
}

// One k-step of the TM x TN register tile: acc[i][j] += a[i] * b[j] as
// TM * TN / 2 packed two-wide FMAs on row pairs (2 i', 2 i' + 1) of column j
// with b[j] in both halves (each half rounds like a scalar fmaf); row pairs in
// serpentine order across columns.
template <int TM, int TN>
__device__ __forceinline__ void outer_product_step(float (&acc)[TM][TN], const float (&a)[TM],
                                                   const float (&b)[TN])
{
#pragma unroll
    for (int j = 0; j < TN; ++j) {
        const float2 bb = make_float2(b[j], b[j]);
#pragma unroll
        for (int ii = 0; ii < TM / 2; ++ii) {
            const int i2 = (j & 1) ? TM / 2 - 1 - ii : ii;
            float2 d = make_float2(acc[2 * i2][j], acc[2 * i2 + 1][j]);
            d = __ffma2_rn(make_float2(a[2 * i2], a[2 * i2 + 1]), bb, d);
            acc[2 * i2][j] = d.x;
            acc[2 * i2 + 1][j] = d.y;
        }
    }
}

// Rows [rank * BM / S, +BM / S) of the cluster's S partial tiles, added in
// rank order and stored to C (masked at M and N).
template <int BM, int BN, bool C_VEC, int S>
__device__ __forceinline__ void cluster_add_parts(const float *part, int M, int N, float *C,
                                                  int m0, int n0, uint32_t rank)
{
    constexpr int kPartPitch = Shape<BM, BN>::kPartPitch;
    constexpr int ROWS = BM / S;
    constexpr int COUNT4 = ROWS * (BN / 4);
    constexpr int ITERS = COUNT4 / kThreads;
    static_assert(COUNT4 % kThreads == 0, "every thread adds whole float4s");
#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
        const int f = (int)threadIdx.x + it * kThreads;
        const int r = (int)rank * ROWS + f / (BN / 4), c = (f % (BN / 4)) * 4;
        const uint32_t local = smem_u32(part + r * kPartPitch + c);
        float4 v[S];
#pragma unroll
        for (int q = 0; q < S; ++q)
            v[q] = S == 1 ? lds128(local) : ld_shared_cluster_v4(mapa_shared(local, (uint32_t)q));
        float4 sum = v[0];
#pragma unroll
        for (int q = 1; q < S; ++q) {
            sum.x += v[q].x;
            sum.y += v[q].y;
            sum.z += v[q].z;
            sum.w += v[q].w;
        }
        const int gm = m0 + r, gn = n0 + c;
        if (gm >= M)
            continue;
        float *crow = C + (size_t)gm * N;
        if constexpr (C_VEC) {
            if (gn < N)
                *reinterpret_cast<float4 *>(crow + gn) = sum;
        } else {
            const float w[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (gn + j < N)
                    crow[gn + j] = w[j];
        }
    }
}

// MUTE (the failure-detection self-test only): thread 0 announces each slice's
// bytes on its barrier but issues no load, so every wait runs out; one CTA per
// SM is enough there, and the register budget that gives keeps it free of spills.
template <int BM, int BN, bool C_VEC, bool MUTE = false>
__global__ void __launch_bounds__(kThreads, MUTE ? 1 : 2)
    sgemm_tma_rect_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB, int M, int N, int K, int kchunk,
                          float *__restrict__ C, int *err, uint64_t wait_limit_ns)
{
    using Sh = Shape<BM, BN>;
    constexpr int TM = Sh::TM, TN = Sh::TN, LDA = Sh::LDA;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int abort_flag;
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char *base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    float *stA = reinterpret_cast<float *>(base + Sh::OFF_ST);
    float *sB = reinterpret_cast<float *>(base + Sh::OFF_B);
    float *sA = reinterpret_cast<float *>(base + Sh::OFF_A);
    uint64_t *full = reinterpret_cast<uint64_t *>(base + Sh::OFF_BAR);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    int tile_m, tile_n;
    tile_of_block((int)blockIdx.x, (M + BM - 1) / BM, (N + BN - 1) / BN, tile_m, tile_n);
    const int m0 = tile_m * BM, n0 = tile_n * BN;
    // 16 x 16 threads: rows rh * 64 + tm * 4 + i, columns ch * 64 + tn * 4 + j;
    // a warp reads 4 distinct 16-byte A fragments and 8 B fragments per load.
    const int tm = (warp >> 1) * 4 + (((lane >> 2) & 1) | ((lane >> 3) & 2));
    const int tn = (warp & 1) * 8 + ((lane & 3) | ((lane >> 1) & 4));
    const int ks_begin = (int)blockIdx.y * (kchunk / BK);
    const int ktiles = max(0, min((K + BK - 1) / BK - ks_begin, kchunk / BK));

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_mbarrier_init();
        abort_flag = 0;
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    __syncthreads();

    int issued = 0, confirmed = 0;
    auto issue = [&](int s) {
        uint64_t *bar = &full[s & 1];
        mbar_arrive_expect_tx(bar, Sh::kSliceBytes);
        if constexpr (!MUTE) {
            tma_load_2d(smem_u32(stA), &tmA, bar, (ks_begin + s) * BK, m0);
            tma_load_2d(smem_u32(sB + (s & 1) * Sh::B_STAGE), &tmB, bar, n0, (ks_begin + s) * BK);
        }
        ++issued;
    };
    // Transpose: thread (r4, q) moves rows 4 r4 + 128 b .. + 3, k 4 q .. 4 q + 3
    // of the staging tile (16-byte chunk c of row r at c ^ (r mod 8)) into the
    // k-major A stage; 64-row tiles need only the threads with r4 < 16.
    const int r4 = warp * 4 + (lane & 3);
    const int q = ((lane >> 3) << 1) | ((lane >> 2) & 1);
    const uint32_t st_base = smem_u32(stA);
    const uint32_t a_dst = smem_u32(sA + (4 * q) * LDA + 4 * r4);
    auto transpose = [&](int s, int stage) {
        if (mbar_wait_bounded(&full[s & 1], (uint32_t)((s >> 1) & 1), wait_limit_ns, &abort_flag)) {
            if (tid == 0 && confirmed == s)
                confirmed = s + 1;
        } else {
            atomicCAS(err, 0, kDevErrTimeout);
            abort_flag = 1;
        }
        if (4 * r4 >= BM)
            return;
#pragma unroll
        for (int b = 0; b < (BM + 127) / 128; ++b) {
            float4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = 128 * b + 4 * r4 + i;
                v[i] = lds128(st_base + (uint32_t)(row * (BK * 4) + ((q ^ (row & 7)) * 16)));
            }
            const uint32_t d = a_dst + (uint32_t)((stage * Sh::A_STAGE + 128 * b) * 4);
            sts128(d + 0 * LDA * 4, v[0].x, v[1].x, v[2].x, v[3].x);
            sts128(d + 1 * LDA * 4, v[0].y, v[1].y, v[2].y, v[3].y);
            sts128(d + 2 * LDA * 4, v[0].z, v[1].z, v[2].z, v[3].z);
            sts128(d + 3 * LDA * 4, v[0].w, v[1].w, v[2].w, v[3].w);
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j)
            acc[i][j] = 0.0f;

    // One k-step of the register tile from A stage `as` and B stage `kt % 2`.
    auto k_step = [&](const float *cA, const float *cB, int k) {
        float a[TM], b[TN];
#pragma unroll
        for (int h = 0; h < TM / 4; ++h) {
            const float4 v = *reinterpret_cast<const float4 *>(cA + k * LDA + h * 64);
            a[h * 4 + 0] = v.x;
            a[h * 4 + 1] = v.y;
            a[h * 4 + 2] = v.z;
            a[h * 4 + 3] = v.w;
        }
#pragma unroll
        for (int h = 0; h < TN / 4; ++h) {
            const float4 v = *reinterpret_cast<const float4 *>(cB + k * BN + h * 64);
            b[h * 4 + 0] = v.x;
            b[h * 4 + 1] = v.y;
            b[h * 4 + 2] = v.z;
            b[h * 4 + 3] = v.w;
        }
        outer_product_step<TM, TN>(acc, a, b);
    };
    if constexpr (Sh::A_STAGES == 1) {
        if (ktiles > 0 && tid == 0)
            issue(0);
        for (int kt = 0; kt < ktiles; ++kt) {
            transpose(kt, 0);
            __syncthreads();  // the A stage holds slice kt; the staging tile is free
            if (tid == 0 && kt + 1 < ktiles && !abort_flag)
                issue(kt + 1);
            const float *cA = sA + tm * 4;
            const float *cB = sB + (kt & 1) * Sh::B_STAGE + tn * 4;
#pragma unroll
            for (int k = 0; k < BK; ++k)
                k_step(cA, cB, k);
            __syncthreads();  // the A stage and B stage kt % 2 are free
        }
    } else {
        // As in sgemm_tma.cu: slice s + 1 is loaded while slice s is multiplied
        // and transposed into the other A stage once slice s's k loop is done.
        if (ktiles > 0) {
            if (tid == 0)
                issue(0);
            transpose(0, 0);
            __syncthreads();
            if (tid == 0 && ktiles > 1 && !abort_flag)
                issue(1);
        }
        for (int kt = 0; kt < ktiles; ++kt) {
            const float *cA = sA + (kt & 1) * Sh::A_STAGE + tm * 4;
            const float *cB = sB + (kt & 1) * Sh::B_STAGE + tn * 4;
            const bool next = kt + 1 < ktiles;
#pragma unroll
            for (int k = 0; k < BK; ++k)
                k_step(cA, cB, k);
            if (next)
                transpose(kt + 1, (kt + 1) & 1);
            __syncthreads();  // stage kt % 2 and the staging tile are free
            if (tid == 0 && kt + 2 < ktiles && !abort_flag)
                issue(kt + 2);
        }
    }
    if (tid == 0 && confirmed < issued) {
        int never = 0;
        for (int s = confirmed; s < issued; ++s)
            mbar_wait_bounded(&full[s & 1], (uint32_t)((s >> 1) & 1), wait_limit_ns, &never);
    }

    // Park the partial tile (the stages are free: the last barrier above).
    float *part = reinterpret_cast<float *>(base);
#pragma unroll
    for (int rh = 0; rh < TM / 4; ++rh)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int ch = 0; ch < TN / 4; ++ch) {
                const float *v = &acc[rh * 4 + i][ch * 4];
                *reinterpret_cast<float4 *>(part + (rh * 64 + tm * 4 + i) * Sh::kPartPitch + ch * 64 +
                                            tn * 4) = make_float4(v[0], v[1], v[2], v[3]);
            }
    const uint32_t rank = blockIdx.y;  // cluster (1, S, 1)
    if (gridDim.y == 1) {
        __syncthreads();
        cluster_add_parts<BM, BN, C_VEC, 1>(part, M, N, C, m0, n0, 0);
        return;
    }
    cluster_sync();
    switch (gridDim.y) {
    case 2: cluster_add_parts<BM, BN, C_VEC, 2>(part, M, N, C, m0, n0, rank); break;
    case 4: cluster_add_parts<BM, BN, C_VEC, 4>(part, M, N, C, m0, n0, rank); break;
    default: cluster_add_parts<BM, BN, C_VEC, 8>(part, M, N, C, m0, n0, rank); break;
    }
    cluster_sync();
}

template <int BM, int BN>
static cudaError_t launch_rect(int M, int N, int K, const float *A, const float *B, float *C,
                               const SimtTma &tma, int splits, int kchunk, bool spread,
                               cudaStream_t stream)
{
    using Sh = Shape<BM, BN>;
    if (!tma.encode_tiled || !tma.err || !sgemm_tma_eligible(M, N, K, A, B, tma.lda, tma.ldb) ||
        (splits != 1 && splits != 2 && splits != 4 && splits != 8) || kchunk % BK != 0 ||
        kchunk <= 0 || (long long)splits * kchunk < K)
        return cudaErrorInvalidValue;
    const long long tiles = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    if (tiles == 0)
        return cudaSuccess;
    if (tiles > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    auto fn = reinterpret_cast<EncodeTiledFn>(tma.encode_tiled);
    CUtensorMap ta, tb;
    if (!encode_f32_map(fn, &ta, A, (uint64_t)M, (uint64_t)K, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B,
                        (uint64_t)tma.lda) ||
        !encode_f32_map(fn, &tb, B, (uint64_t)K, (uint64_t)N, BN, BK, CU_TENSOR_MAP_SWIZZLE_NONE,
                        (uint64_t)tma.ldb))
        return cudaErrorInvalidValue;
    const bool c_vec = N % 4 == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0;
    auto kernel = tma.mute ? (c_vec ? sgemm_tma_rect_kernel<BM, BN, true, true>
                                    : sgemm_tma_rect_kernel<BM, BN, false, true>)
                           : (c_vec ? sgemm_tma_rect_kernel<BM, BN, true>
                                    : sgemm_tma_rect_kernel<BM, BN, false>);
    static std::atomic<uint64_t> done[4] = {{0}, {0}, {0}, {0}};
    const cudaError_t e =
        set_smem_limit_once(kernel, kSpreadSmem, done[(tma.mute ? 2 : 0) + (c_vec ? 0 : 1)]);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, (unsigned)splits, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = spread ? kSpreadSmem : Sh::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)splits;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, ta, tb, M, N, K, kchunk, C, tma.err,
                              tma.wait_limit_ns);
}

} // namespace simt_tma_rect

cudaError_t launch_sgemm_f32_tma_rect(SimtTile tile, int M, int N, int K, const float *A,
                                      const float *B, float *C, const SimtTma &tma, int splits,
                                      int kchunk, bool spread, cudaStream_t stream)
{
    using namespace simt_tma_rect;
    if (tile.m == 256 && tile.n == 64)
        return launch_rect<256, 64>(M, N, K, A, B, C, tma, splits, kchunk, spread, stream);
    if (tile.m == 64 && tile.n == 256)
        return launch_rect<64, 256>(M, N, K, A, B, C, tma, splits, kchunk, spread, stream);
    return cudaErrorInvalidValue;
}

} // namespace rtm
