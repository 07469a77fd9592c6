// SIMT FP32 register-tiled product C = A.B, 128 x 128 C tiles, with the
// shared-memory level fed by the tensor-memory-access (TMA) unit.
//
// The register level and the shared-memory layouts are those of the
// cp.async kernel (sgemm_simt.cu): 16 x 16 threads, 8 x 8 accumulators per
// thread as 2 x 2 sub-blocks of 4 x 4 spaced 64 apart, 32-deep K slices, A
// k-major with rows padded to 132 floats, B as stored; per k, 4 LDS.128 feed
// 64 FMAs, here as 32 packed two-wide FMAs ("理解 Register Tiling", section
// "关键循环：为什么省了 Shared Memory 读取？"; "寄存器Tiling跨架构解析",
// sections 1.1 and 6.3 on staging K slices through shared memory).
//
// What changes is who moves the data. In the cp.async kernel every thread
// issues 20 copies per slice (16 four-byte copies that transpose A, 4
// sixteen-byte copies of B) and computes their addresses: on GB300 that is
// about 110 of the 2340 instructions a warp issues per slice, in a loop bound
// by instruction issue. Here one thread issues two TMA loads per slice — a
// 128 m x 32 k box of A (row-major, 128-byte swizzle) into a staging tile and
// a 32 k x 128 n box of B straight into the B stage — and every thread then
// moves one 4 x 4 block of A from the staging tile into the k-major A stage
// with 4 LDS.128 and 4 STS.128 (a transpose in registers). The TMA unit
// zero-fills rows, columns and K beyond the matrices, so edge tiles and the
// last, partial slice need no predicated copies; stores to C are masked.
//
// Pipeline (two A and B stages, one staging tile, one CTA barrier per slice):
// slice s+1 is loaded while slice s is multiplied; at the end of slice s's
// k loop every thread waits for slice s+1's loads (an mbarrier with the
// byte count of both boxes) and transposes its block, the CTA barrier then
// frees the staging tile and the stage slice s used, and thread 0 issues
// slice s+2 into them. Every mbarrier wait is bounded; a wait that gives up
// records GEMM_ERR_TIMEOUT in the device error word and raises the CTA's
// abort flag, so every thread still reaches every barrier and the kernel
// ends; once the flag is up thread 0 issues no further slice (a barrier whose
// phase never completed must not be armed again).
//
// Requirements (checked by the launcher): K % 4 == 0 and N % 4 == 0 (TMA row
// strides are multiples of 16 bytes), A and B 16-byte aligned. The sum over k
// runs in the same order with the same rounding as the cp.async kernel, so
// the two give the same bits.
#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"
#include "simt_tma_common.cuh"

namespace rtm {
namespace simt_tma {

constexpr int kThreads = 256;
constexpr int BM = 128, BN = 128, BK = 32;
constexpr int LDA = BM + 4;          // k-major A rows, padded (conflict-free stores and reads)
constexpr int A_STAGE = BK * LDA;    // floats per A stage
constexpr int B_STAGE = BK * BN;     // floats per B stage
// Tile-rows per L2 group. At 4096^3 (32 x 32 tiles, 304 CTAs resident) the
// DRAM reads per launch measured 346 MB with groups of 8 rows, 281 MB with
// 16 and 506 MB with 32 (A and B hold 134 MB), at the same speed.
constexpr int kGroupM = 16;
// Shared-memory layout in bytes from a 1024-byte-aligned base (the 128-byte
// swizzle repeats every 1024 bytes): staging tile, two B stages, two A
// stages, two mbarriers.
constexpr int OFF_ST = 0;
constexpr int OFF_B = BM * BK * 4;
constexpr int OFF_A = OFF_B + 2 * B_STAGE * 4;
constexpr int OFF_BAR = OFF_A + 2 * A_STAGE * 4;
constexpr int SMEM_BYTES = OFF_BAR + 16 + 1024;  // + room to align the base
constexpr uint32_t kSliceBytes = (BM * BK + BK * BN) * 4;
constexpr int kSpreadSmem = 120 * 1024;  // more than half of an SM's 228 KB

using simt_tma_common::EncodeTiledFn;
using simt_tma_common::encode_f32_map;
using simt_tma_common::lds128;
using simt_tma_common::sts128;

__device__ __forceinline__ void tile_of_block(int bid, int tiles_m, int tiles_n, int &tile_m,
                                              int &tile_n)
{
    simt_tma_common::grouped_tile<kGroupM>(bid, tiles_m, tiles_n, tile_m, tile_n);
}

// One k-step of the 8 x 8 register tile: acc[i][j] += a[i] * b[j], as 32
// packed two-wide FMAs (fma.rn.f32x2) on pairs of rows (2 i', 2 i' + 1) of
// one column j, with b[j] in both halves; each half rounds exactly like a
// scalar fmaf, so every accumulator sees the same operations in the same
// order as the scalar loop. Columns in order, row pairs in serpentine
// order. On GB300 4096^3: 2.255 ms with scalar FFMA, 2.141 ms packed (pairs
// along n with a[i] in both halves: 2.152 ms); half the FMA instructions
// leave issue slots to the loads and the transpose.
__device__ __forceinline__ void outer_product_step(float (&acc)[8][8], const float (&a)[8],
                                                   const float (&b)[8])
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float2 bb = make_float2(b[j], b[j]);
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
            const int i2 = (j & 1) ? 3 - ii : ii;
            float2 d = make_float2(acc[2 * i2][j], acc[2 * i2 + 1][j]);
            d = __ffma2_rn(make_float2(a[2 * i2], a[2 * i2 + 1]), bb, d);
            acc[2 * i2][j] = d.x;
            acc[2 * i2 + 1][j] = d.y;
        }
    }
}

// MUTE (the failure-detection self-test only): thread 0 announces each slice's
// bytes on its barrier but issues no load, so every wait runs out.
template <bool C_VEC, bool MUTE = false>
__global__ void __launch_bounds__(kThreads, 2)
    sgemm_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     int M, int N, int K, float *__restrict__ C, int *err, uint64_t wait_limit_ns)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int abort_flag;
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char *base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    float *stA = reinterpret_cast<float *>(base + OFF_ST);  // [BM][BK], 128-byte swizzle
    float *sB = reinterpret_cast<float *>(base + OFF_B);    // [2][BK][BN]
    float *sA = reinterpret_cast<float *>(base + OFF_A);    // [2][BK][LDA], k-major
    uint64_t *full = reinterpret_cast<uint64_t *>(base + OFF_BAR);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    int tile_m, tile_n;
    tile_of_block(blockIdx.x, (M + BM - 1) / BM, (N + BN - 1) / BN, tile_m, tile_n);
    const int m0 = tile_m * BM, n0 = tile_n * BN;
    // Thread (tm, tn) of the 16 x 16 grid, the cp.async kernel's lane map.
    const int tm = (warp >> 1) * 4 + (((lane >> 2) & 1) | ((lane >> 3) & 2));
    const int tn = (warp & 1) * 8 + ((lane & 3) | ((lane >> 1) & 4));
    const int ktiles = (K + BK - 1) / BK;

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_mbarrier_init();
        abort_flag = 0;
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    __syncthreads();

    // Thread 0: slice s of A into the staging tile, of B into B stage s % 2.
    int issued = 0, confirmed = 0;  // thread 0's count of slices issued / seen landed
    auto issue = [&](int s) {
        uint64_t *bar = &full[s & 1];
        mbar_arrive_expect_tx(bar, kSliceBytes);
        if constexpr (!MUTE) {
            tma_load_2d(smem_u32(stA), &tmA, bar, s * BK, m0);
            tma_load_2d(smem_u32(sB + (s & 1) * B_STAGE), &tmB, bar, n0, s * BK);
        }
        ++issued;
    };

    // Transpose: thread (r4, q) moves rows 4 r4 .. +3, k 4 q .. +3 of the
    // staging tile (16-byte chunk c of row r sits at c ^ (r % 8)) into the
    // k-major stage, one STS.128 per k. Quarter-warps hold two q and four r4,
    // so the stores hit 8 distinct 16-byte bank groups (row pitch 132 floats).
    const int r4 = warp * 4 + (lane & 3);
    const int q = ((lane >> 3) << 1) | ((lane >> 2) & 1);
    const uint32_t st_base = smem_u32(stA);
    const uint32_t a_dst = smem_u32(sA + (4 * q) * LDA + 4 * r4);
    auto transpose = [&](int s) {
        if (mbar_wait_bounded(&full[s & 1], (uint32_t)((s >> 1) & 1), wait_limit_ns, &abort_flag)) {
            if (tid == 0 && confirmed == s)
                confirmed = s + 1;
        } else {
            atomicCAS(err, 0, kDevErrTimeout);
            abort_flag = 1;
        }
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = 4 * r4 + i;
            v[i] = lds128(st_base + (uint32_t)(row * (BK * 4) + ((q ^ (row & 7)) * 16)));
        }
        const uint32_t d = a_dst + (uint32_t)((s & 1) * A_STAGE * 4);
        sts128(d + 0 * LDA * 4, v[0].x, v[1].x, v[2].x, v[3].x);
        sts128(d + 1 * LDA * 4, v[0].y, v[1].y, v[2].y, v[3].y);
        sts128(d + 2 * LDA * 4, v[0].z, v[1].z, v[2].z, v[3].z);
        sts128(d + 3 * LDA * 4, v[0].w, v[1].w, v[2].w, v[3].w);
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j)
            acc[i][j] = 0.0f;

    if (tid == 0)
        issue(0);
    transpose(0);
    __syncthreads();
    if (tid == 0 && ktiles > 1 && !abort_flag)
        issue(1);

    for (int kt = 0; kt < ktiles; ++kt) {
        const float *cA = sA + (kt & 1) * A_STAGE + tm * 4;
        const float *cB = sB + (kt & 1) * B_STAGE + tn * 4;
        const bool next = kt + 1 < ktiles;
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float a[8], b[8];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float4 v = *reinterpret_cast<const float4 *>(cA + k * LDA + h * 64);
                a[h * 4 + 0] = v.x;
                a[h * 4 + 1] = v.y;
                a[h * 4 + 2] = v.z;
                a[h * 4 + 3] = v.w;
            }
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const float4 v = *reinterpret_cast<const float4 *>(cB + k * BN + p * 64);
                b[p * 4 + 0] = v.x;
                b[p * 4 + 1] = v.y;
                b[p * 4 + 2] = v.z;
                b[p * 4 + 3] = v.w;
            }
            outer_product_step(acc, a, b);
            if (k == BK - 1 && next)
                transpose(kt + 1);
        }
        __syncthreads();  // stage kt and the staging tile are free
        if (tid == 0 && kt + 2 < ktiles && !abort_flag)
            issue(kt + 2);
    }

    // Only after a wait gave up can loads still be in flight: thread 0 waits
    // for them (bounded, without the abort shortcut) before the CTA leaves.
    if (tid == 0 && confirmed < issued) {
        int never = 0;
        for (int s = confirmed; s < issued; ++s)
            mbar_wait_bounded(&full[s & 1], (uint32_t)((s >> 1) & 1), wait_limit_ns, &never);
    }

    // Epilogue: masked stores, 128-bit where C rows allow it.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gm = m0 + h * 64 + tm * 4 + i;
            if (gm >= M)
                continue;
            float *crow = C + (size_t)gm * N;
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const int gn = n0 + p * 64 + tn * 4;
                const float *v = &acc[h * 4 + i][p * 4];
                if constexpr (C_VEC) {
                    if (gn < N)
                        *reinterpret_cast<float4 *>(crow + gn) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (gn + j < N)
                            crow[gn + j] = v[j];
                }
            }
        }
    }
}

// K split over the S CTAs of a thread-block cluster, as the cp.async kernel's
// cluster mode (sgemm_simt.cu) but with this file's TMA-fed, packed-FMA loop:
// grid (tiles, S), cluster (1, S, 1); CTA y of a cluster multiplies K-slices
// [y * kchunk, +kchunk) of tile tile_first + blockIdx.x, parks its partial tile
// in its own shared memory (rows padded to BN + 4 floats), and after a cluster
// barrier adds rows [y * BM / S, +BM / S) of the S partials, read through
// distributed shared memory in rank order (the same sum on every call), and
// stores them. A second barrier keeps every partial alive until it is read.
constexpr int kPartPitch = BN + 4;
static_assert(BM * kPartPitch * 4 <= OFF_BAR, "the partial tile fits below the barriers");

template <bool C_VEC, int S>
__device__ __forceinline__ void cluster_add_parts(const float *part, int M, int N, float *C,
                                                  int m0, int n0, uint32_t rank)
{
    constexpr int ROWS = BM / S;
    constexpr int COUNT4 = ROWS * (BN / 4);
    constexpr int ITERS = COUNT4 / kThreads;
    static_assert(COUNT4 % kThreads == 0, "every thread adds whole float4s");
    float4 v[ITERS][S];
#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
        const int f = (int)threadIdx.x + it * kThreads;
        const int r = (int)rank * ROWS + f / (BN / 4), c = (f % (BN / 4)) * 4;
        const uint32_t local = smem_u32(part + r * kPartPitch + c);
#pragma unroll
        for (int q = 0; q < S; ++q)
            v[it][q] = ld_shared_cluster_v4(mapa_shared(local, (uint32_t)q));
    }
#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
        float4 sum = v[it][0];
#pragma unroll
        for (int q = 1; q < S; ++q) {
            sum.x += v[it][q].x;
            sum.y += v[it][q].y;
            sum.z += v[it][q].z;
            sum.w += v[it][q].w;
        }
        const int f = (int)threadIdx.x + it * kThreads;
        const int gm = m0 + (int)rank * ROWS + f / (BN / 4), gn = n0 + (f % (BN / 4)) * 4;
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

// MUTE (the self-test): as in sgemm_tma_kernel; one CTA per SM is enough
// there, and the register budget that gives keeps the variant free of spills.
template <bool C_VEC, bool MUTE = false>
__global__ void __launch_bounds__(kThreads, MUTE ? 1 : 2)
    sgemm_tma_cluster_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB, int M, int N, int K,
                             int kchunk, int tile_first, float *__restrict__ C, int *err,
                             uint64_t wait_limit_ns)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int abort_flag;
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char *base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    float *stA = reinterpret_cast<float *>(base + OFF_ST);
    float *sB = reinterpret_cast<float *>(base + OFF_B);
    float *sA = reinterpret_cast<float *>(base + OFF_A);
    uint64_t *full = reinterpret_cast<uint64_t *>(base + OFF_BAR);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    int tile_m, tile_n;
    tile_of_block((int)blockIdx.x + tile_first, (M + BM - 1) / BM, (N + BN - 1) / BN, tile_m,
                  tile_n);
    const int m0 = tile_m * BM, n0 = tile_n * BN;
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
        mbar_arrive_expect_tx(bar, kSliceBytes);
        if constexpr (!MUTE) {
            tma_load_2d(smem_u32(stA), &tmA, bar, (ks_begin + s) * BK, m0);
            tma_load_2d(smem_u32(sB + (s & 1) * B_STAGE), &tmB, bar, n0, (ks_begin + s) * BK);
        }
        ++issued;
    };
    const int r4 = warp * 4 + (lane & 3);
    const int q = ((lane >> 3) << 1) | ((lane >> 2) & 1);
    const uint32_t st_base = smem_u32(stA);
    const uint32_t a_dst = smem_u32(sA + (4 * q) * LDA + 4 * r4);
    auto transpose = [&](int s) {
        if (mbar_wait_bounded(&full[s & 1], (uint32_t)((s >> 1) & 1), wait_limit_ns, &abort_flag)) {
            if (tid == 0 && confirmed == s)
                confirmed = s + 1;
        } else {
            atomicCAS(err, 0, kDevErrTimeout);
            abort_flag = 1;
        }
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = 4 * r4 + i;
            v[i] = lds128(st_base + (uint32_t)(row * (BK * 4) + ((q ^ (row & 7)) * 16)));
        }
        const uint32_t d = a_dst + (uint32_t)((s & 1) * A_STAGE * 4);
        sts128(d + 0 * LDA * 4, v[0].x, v[1].x, v[2].x, v[3].x);
        sts128(d + 1 * LDA * 4, v[0].y, v[1].y, v[2].y, v[3].y);
        sts128(d + 2 * LDA * 4, v[0].z, v[1].z, v[2].z, v[3].z);
        sts128(d + 3 * LDA * 4, v[0].w, v[1].w, v[2].w, v[3].w);
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j)
            acc[i][j] = 0.0f;

    if (ktiles > 0) {
        if (tid == 0)
            issue(0);
        transpose(0);
        __syncthreads();
        if (tid == 0 && ktiles > 1 && !abort_flag)
            issue(1);
    }
    for (int kt = 0; kt < ktiles; ++kt) {
        const float *cA = sA + (kt & 1) * A_STAGE + tm * 4;
        const float *cB = sB + (kt & 1) * B_STAGE + tn * 4;
        const bool next = kt + 1 < ktiles;
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float a[8], b[8];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float4 v = *reinterpret_cast<const float4 *>(cA + k * LDA + h * 64);
                a[h * 4 + 0] = v.x;
                a[h * 4 + 1] = v.y;
                a[h * 4 + 2] = v.z;
                a[h * 4 + 3] = v.w;
            }
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const float4 v = *reinterpret_cast<const float4 *>(cB + k * BN + p * 64);
                b[p * 4 + 0] = v.x;
                b[p * 4 + 1] = v.y;
                b[p * 4 + 2] = v.z;
                b[p * 4 + 3] = v.w;
            }
            outer_product_step(acc, a, b);
            if (k == BK - 1 && next)
                transpose(kt + 1);
        }
        __syncthreads();
        if (tid == 0 && kt + 2 < ktiles && !abort_flag)
            issue(kt + 2);
    }
    if (tid == 0 && confirmed < issued) {
        int never = 0;
        for (int s = confirmed; s < issued; ++s)
            mbar_wait_bounded(&full[s & 1], (uint32_t)((s >> 1) & 1), wait_limit_ns, &never);
    }

    // Park the partial tile (the stages are free: the last barrier above).
    float *part = reinterpret_cast<float *>(base);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const float *v = &acc[h * 4 + i][p * 4];
                *reinterpret_cast<float4 *>(part + (h * 64 + tm * 4 + i) * kPartPitch + p * 64 +
                                            tn * 4) = make_float4(v[0], v[1], v[2], v[3]);
            }
    cluster_sync();
    const uint32_t rank = blockIdx.y;  // cluster (1, S, 1)
    switch (gridDim.y) {
    case 2: cluster_add_parts<C_VEC, 2>(part, M, N, C, m0, n0, rank); break;
    case 4: cluster_add_parts<C_VEC, 4>(part, M, N, C, m0, n0, rank); break;
    case 8: cluster_add_parts<C_VEC, 8>(part, M, N, C, m0, n0, rank); break;
    default: cluster_add_parts<C_VEC, 1>(part, M, N, C, m0, n0, rank); break;
    }
    cluster_sync();
}

// Stream-K ("寄存器Tiling跨架构解析", sections 2.4 and 7.2: work per block
// and how many blocks keep the SMs busy). The product's tiles x K-slices
// iterations I are cut into gridDim.x equal ranges, one per CTA: CTA c takes
// iterations [b(c), b(c + 1)) with b(c) = floor(c I / G), where iteration g is
// K-slice g % ktiles of tile g / ktiles (grouped raster order). The TMA
// pipeline runs straight across tile boundaries. When a CTA's range ends a
// tile, or its range ends, the accumulators go out: a tile the CTA computed
// whole goes to C, a part of a tile to slot c + t of the workspace W (a dense
// BM x BN tile; c + t is unique because the tiles of CTA c are never beyond
// those of CTA c + 1). sgemm_streamk_fixup_kernel then adds each split tile's
// parts in increasing c (increasing k), so the result repeats bit for bit.
template <bool C_VEC>
__global__ void __launch_bounds__(kThreads, 2)
    sgemm_tma_streamk_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB, int M, int N, int K,
                             float *__restrict__ C, float *__restrict__ W, int *err,
                             uint64_t wait_limit_ns)
{
    grid_launch_dependents();  // the fixup may launch; it waits for this grid to finish
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int abort_flag;
    __shared__ int issued, confirmed;  // thread 0's count of slices issued / seen landed
    __shared__ int it_ks, it_m0, it_n0, it_tile;  // thread 0: the next slice to issue
    // This CTA's range, written once by thread 0 and read where it is used
    // (volatile), so that none of it holds a register across the FMA loop.
    __shared__ int sk_n, sk_t0, sk_ks0, sk_ktiles, sk_tiles_m, sk_tiles_n;
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char *base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    float *stA = reinterpret_cast<float *>(base + OFF_ST);
    float *sB = reinterpret_cast<float *>(base + OFF_B);
    float *sA = reinterpret_cast<float *>(base + OFF_A);
    uint64_t *full = reinterpret_cast<uint64_t *>(base + OFF_BAR);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int tm = (warp >> 1) * 4 + (((lane >> 2) & 1) | ((lane >> 3) & 2));
    const int tn = (warp & 1) * 8 + ((lane & 3) | ((lane >> 1) & 4));

    if (tid == 0) {
        const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
        const int ktiles = (K + BK - 1) / BK;
        const long long iters = (long long)tiles_m * tiles_n * ktiles;
        const long long g0 = (long long)blockIdx.x * iters / gridDim.x;
        const int t0 = (int)(g0 / ktiles);
        sk_n = (int)((long long)(blockIdx.x + 1) * iters / gridDim.x - g0);
        sk_t0 = t0;
        sk_ks0 = (int)(g0 % ktiles);
        sk_ktiles = ktiles;
        sk_tiles_m = tiles_m;
        sk_tiles_n = tiles_n;
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_mbarrier_init();
        abort_flag = 0;
        issued = 0;
        confirmed = 0;
        int tmi, tni;
        tile_of_block(t0, tiles_m, tiles_n, tmi, tni);
        it_tile = t0;
        it_ks = sk_ks0;
        it_m0 = tmi * BM;
        it_n0 = tni * BN;
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    __syncthreads();
    auto shared_int = [](const int &v) { return *reinterpret_cast<const volatile int *>(&v); };
    const int n = shared_int(sk_n);

    // Thread 0: slice s of this CTA's range into stage s % 2. Its position
    // (tile, K-slice) advances by one per call and lives in shared memory, so
    // no division runs per slice and no register is taken from the loop.
    auto issue = [&](int s) {
        const int ks = it_ks;
        uint64_t *bar = &full[s & 1];
        mbar_arrive_expect_tx(bar, kSliceBytes);
        tma_load_2d(smem_u32(stA), &tmA, bar, ks * BK, it_m0);
        tma_load_2d(smem_u32(sB + (s & 1) * B_STAGE), &tmB, bar, it_n0, ks * BK);
        ++issued;
        if (ks + 1 == sk_ktiles) {
            int tmi, tni;
            tile_of_block(++it_tile, sk_tiles_m, sk_tiles_n, tmi, tni);
            it_m0 = tmi * BM;
            it_n0 = tni * BN;
            it_ks = 0;
        } else {
            it_ks = ks + 1;
        }
    };
    const int r4 = warp * 4 + (lane & 3);
    const int q = ((lane >> 3) << 1) | ((lane >> 2) & 1);
    const uint32_t st_base = smem_u32(stA);
    const uint32_t a_dst = smem_u32(sA + (4 * q) * LDA + 4 * r4);
    auto transpose = [&](int s) {
        if (mbar_wait_bounded(&full[s & 1], (uint32_t)((s >> 1) & 1), wait_limit_ns, &abort_flag)) {
            if (tid == 0 && confirmed == s)
                confirmed = s + 1;
        } else {
            atomicCAS(err, 0, kDevErrTimeout);
            abort_flag = 1;
        }
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = 4 * r4 + i;
            v[i] = lds128(st_base + (uint32_t)(row * (BK * 4) + ((q ^ (row & 7)) * 16)));
        }
        const uint32_t d = a_dst + (uint32_t)((s & 1) * A_STAGE * 4);
        sts128(d + 0 * LDA * 4, v[0].x, v[1].x, v[2].x, v[3].x);
        sts128(d + 1 * LDA * 4, v[0].y, v[1].y, v[2].y, v[3].y);
        sts128(d + 2 * LDA * 4, v[0].z, v[1].z, v[2].z, v[3].z);
        sts128(d + 3 * LDA * 4, v[0].w, v[1].w, v[2].w, v[3].w);
    };

    if (n > 0) {
        if (tid == 0)
            issue(0);
        transpose(0);
        __syncthreads();
        if (tid == 0 && n > 1 && !abort_flag)
            issue(1);
    }
    // Tile segments of the range: [s, s + len) is K-slices ks0 .. ks0 + len - 1
    // of one tile. The inner loop is the plain kernel's slice loop.
    for (int s = 0, t = shared_int(sk_t0), ks0 = shared_int(sk_ks0); s < n; ++t, ks0 = 0) {
        const int ktiles = shared_int(sk_ktiles);
        const int len = min(n - s, ktiles - ks0);
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                acc[i][j] = 0.0f;
        for (const int send = s + len; s < send; ++s) {
            const float *cA = sA + (s & 1) * A_STAGE + tm * 4;
            const float *cB = sB + (s & 1) * B_STAGE + tn * 4;
            const bool next = s + 1 < n;
#pragma unroll
            for (int k = 0; k < BK; ++k) {
                float a[8], b[8];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 v = *reinterpret_cast<const float4 *>(cA + k * LDA + h * 64);
                    a[h * 4 + 0] = v.x;
                    a[h * 4 + 1] = v.y;
                    a[h * 4 + 2] = v.z;
                    a[h * 4 + 3] = v.w;
                }
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const float4 v = *reinterpret_cast<const float4 *>(cB + k * BN + p * 64);
                    b[p * 4 + 0] = v.x;
                    b[p * 4 + 1] = v.y;
                    b[p * 4 + 2] = v.z;
                    b[p * 4 + 3] = v.w;
                }
                outer_product_step(acc, a, b);
                if (k == BK - 1 && next)
                    transpose(s + 1);
            }
            __syncthreads();  // stage s % 2 and the staging tile are free
            if (tid == 0 && s + 2 < n && !abort_flag)
                issue(s + 2);
        }
        // The segment's accumulators: a whole tile to C, a part to its slot.
        int tmi, tni;
        tile_of_block(t, shared_int(sk_tiles_m), shared_int(sk_tiles_n), tmi, tni);
        const bool whole = ks0 == 0 && len == shared_int(sk_ktiles);
        float *slot = W + (size_t)(blockIdx.x + t) * (BM * BN);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = h * 64 + tm * 4 + i;
                const int gm = tmi * BM + r;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int cc = p * 64 + tn * 4;
                    const float *v = &acc[h * 4 + i][p * 4];
                    if (!whole) {
                        *reinterpret_cast<float4 *>(slot + r * BN + cc) =
                            make_float4(v[0], v[1], v[2], v[3]);
                    } else if (gm < M) {
                        const int gn = tni * BN + cc;
                        float *crow = C + (size_t)gm * N;
                        if constexpr (C_VEC) {
                            if (gn < N)
                                *reinterpret_cast<float4 *>(crow + gn) =
                                    make_float4(v[0], v[1], v[2], v[3]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                if (gn + j < N)
                                    crow[gn + j] = v[j];
                        }
                    }
                }
            }
    }
    if (tid == 0 && confirmed < issued) {
        int never = 0;
        for (int s = confirmed; s < issued; ++s)
            mbar_wait_bounded(&full[s & 1], (uint32_t)((s >> 1) & 1), wait_limit_ns, &never);
    }
}

// The CTA of the stream-K grid (ctas CTAs over `iters` iterations) whose
// range holds iteration g.
__device__ __forceinline__ long long streamk_cta_of(long long g, long long iters, int ctas)
{
    return ((g + 1) * ctas - 1) / iters;
}

// Tiles split between CTAs c0 < ... < c1 get C = W[c0 + t] + ... + W[c1 + t],
// added in that order; tiles computed whole are left alone. Grid (tiles,
// kFixupParts): CTA (t, y) owns rows y * BM / kFixupParts .. of tile t, one
// float4 per thread, and loads up to 8 parts before adding them, so the
// fixup runs at the speed of its loads rather than one L2 round trip per part.
constexpr int kFixupParts = BM * BN / 4 / kThreads;  // 16: one float4 per thread

template <bool C_VEC>
__global__ void __launch_bounds__(kThreads)
    sgemm_streamk_fixup_kernel(const float *__restrict__ W, float *__restrict__ C, int M, int N,
                               int K, int ctas)
{
    grid_dependency_wait();  // the stream-K grid has finished and its stores are visible
    const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
    const int ktiles = (K + BK - 1) / BK;
    const long long iters = (long long)tiles_m * tiles_n * ktiles;
    const int t = (int)blockIdx.x;
    const long long c0 = streamk_cta_of((long long)t * ktiles, iters, ctas);
    const long long c1 = streamk_cta_of((long long)t * ktiles + ktiles - 1, iters, ctas);
    if (c0 == c1)
        return;
    int tmi, tni;
    tile_of_block(t, tiles_m, tiles_n, tmi, tni);
    const int f = (int)blockIdx.y * kThreads + (int)threadIdx.x;  // float4 index in the tile
    const int r = f / (BN / 4), cc = (f % (BN / 4)) * 4;
    const size_t off = (size_t)r * BN + cc;
    auto part = [&](long long c) {
        return *reinterpret_cast<const float4 *>(W + (size_t)(c + t) * (BM * BN) + off);
    };
    float4 sum = part(c0);
    for (long long c = c0 + 1; c <= c1; c += 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (c + u <= c1)
                v[u] = part(c + u);
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (c + u <= c1) {
                sum.x += v[u].x;
                sum.y += v[u].y;
                sum.z += v[u].z;
                sum.w += v[u].w;
            }
    }
    const int gm = tmi * BM + r, gn = tni * BN + cc;
    if (gm >= M)
        return;
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

} // namespace simt_tma

bool sgemm_tma_eligible(int M, int N, int K, const float *A, const float *B, int64_t lda,
                        int64_t ldb)
{
    (void)M;
    return (lda ? lda : K) % 4 == 0 && (ldb ? ldb : N) % 4 == 0 &&
           (reinterpret_cast<uintptr_t>(A) & 15) == 0 && (reinterpret_cast<uintptr_t>(B) & 15) == 0;
}

cudaError_t launch_sgemm_f32_tma(int M, int N, int K, const float *A, const float *B, float *C,
                                 const SimtTma &tma, long long tile_count, cudaStream_t stream,
                                 bool mute)
{
    using namespace simt_tma;
    if (!tma.encode_tiled || !tma.err || !sgemm_tma_eligible(M, N, K, A, B, tma.lda, tma.ldb))
        return cudaErrorInvalidValue;
    const long long all_tiles = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const long long tiles = tile_count < 0 || tile_count > all_tiles ? all_tiles : tile_count;
    if (tiles > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    if (tiles == 0)
        return cudaSuccess;
    auto fn = reinterpret_cast<EncodeTiledFn>(tma.encode_tiled);
    CUtensorMap ta, tb;
    if (!encode_f32_map(fn, &ta, A, (uint64_t)M, (uint64_t)K, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B,
                        (uint64_t)tma.lda) ||
        !encode_f32_map(fn, &tb, B, (uint64_t)K, (uint64_t)N, BN, BK, CU_TENSOR_MAP_SWIZZLE_NONE,
                        (uint64_t)tma.ldb))
        return cudaErrorInvalidValue;
    const bool c_vec = N % 4 == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0;
    // Muted (the self-test) or not, the epilogue stores whatever C's alignment allows.
    const bool m = mute || tma.mute;
    auto kernel = m ? (c_vec ? sgemm_tma_kernel<true, true> : sgemm_tma_kernel<false, true>)
                    : (c_vec ? sgemm_tma_kernel<true> : sgemm_tma_kernel<false>);
    static std::atomic<uint64_t> done[4] = {{0}, {0}, {0}, {0}};
    const cudaError_t e = set_smem_limit_once(kernel, SMEM_BYTES, done[(m ? 2 : 0) + (c_vec ? 0 : 1)]);
    if (e != cudaSuccess)
        return e;
    kernel<<<(unsigned)tiles, kThreads, SMEM_BYTES, stream>>>(ta, tb, M, N, K, C, tma.err,
                                                               tma.wait_limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_sgemm_f32_tma_cluster(int M, int N, int K, const float *A, const float *B,
                                         float *C, const SimtTma &tma, int splits, int kchunk,
                                         bool spread, long long tile_first, long long tile_count,
                                         cudaStream_t stream)
{
    using namespace simt_tma;
    if (!tma.encode_tiled || !tma.err || !sgemm_tma_eligible(M, N, K, A, B, tma.lda, tma.ldb) ||
        (splits != 1 && splits != 2 && splits != 4 && splits != 8) || kchunk % BK != 0 ||
        (long long)splits * kchunk < K)
        return cudaErrorInvalidValue;
    const long long all_tiles = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    if (all_tiles > 0x7fffffffLL || tile_first < 0 || tile_first > all_tiles)
        return cudaErrorInvalidValue;
    const long long tiles = tile_count < 0 || tile_first + tile_count > all_tiles
                                ? all_tiles - tile_first
                                : tile_count;
    if (tiles == 0)
        return cudaSuccess;
    auto fn = reinterpret_cast<EncodeTiledFn>(tma.encode_tiled);
    CUtensorMap ta, tb;
    if (!encode_f32_map(fn, &ta, A, (uint64_t)M, (uint64_t)K, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B,
                        (uint64_t)tma.lda) ||
        !encode_f32_map(fn, &tb, B, (uint64_t)K, (uint64_t)N, BN, BK, CU_TENSOR_MAP_SWIZZLE_NONE,
                        (uint64_t)tma.ldb))
        return cudaErrorInvalidValue;
    const bool c_vec = N % 4 == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0;
    auto kernel = tma.mute ? (c_vec ? sgemm_tma_cluster_kernel<true, true>
                                    : sgemm_tma_cluster_kernel<false, true>)
                           : (c_vec ? sgemm_tma_cluster_kernel<true> : sgemm_tma_cluster_kernel<false>);
    static std::atomic<uint64_t> done[4] = {{0}, {0}, {0}, {0}};
    const cudaError_t e =
        set_smem_limit_once(kernel, kSpreadSmem, done[(tma.mute ? 2 : 0) + (c_vec ? 0 : 1)]);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, (unsigned)splits, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = spread ? kSpreadSmem : SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)splits;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, ta, tb, M, N, K, kchunk, (int)tile_first, C, tma.err,
                              tma.wait_limit_ns);
}

int64_t sgemm_streamk_workspace_floats(int M, int N, int ctas)
{
    const long long tiles = (long long)((M + simt_tma::BM - 1) / simt_tma::BM) *
                            ((N + simt_tma::BN - 1) / simt_tma::BN);
    return (tiles + ctas - 1) * (int64_t)(simt_tma::BM * simt_tma::BN);
}

cudaError_t launch_sgemm_f32_streamk(int M, int N, int K, const float *A, const float *B, float *C,
                                     const SimtTma &tma, int ctas, bool spread, float *workspace,
                                     cudaStream_t stream)
{
    using namespace simt_tma;
    if (!tma.encode_tiled || !tma.err || !sgemm_tma_eligible(M, N, K, A, B, tma.lda, tma.ldb) || ctas < 1 ||
        !workspace || (reinterpret_cast<uintptr_t>(workspace) & 15) != 0)
        return cudaErrorInvalidValue;
    const long long tiles = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    if (tiles > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    // Every CTA gets at least one iteration (the fixup adds the parts of the
    // CTAs c0 .. c1 that share a tile, so none of them may be empty).
    const long long iters = tiles * ((K + BK - 1) / BK);
    if (ctas > iters)
        ctas = (int)iters;
    auto fn = reinterpret_cast<EncodeTiledFn>(tma.encode_tiled);
    CUtensorMap ta, tb;
    if (!encode_f32_map(fn, &ta, A, (uint64_t)M, (uint64_t)K, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B,
                        (uint64_t)tma.lda) ||
        !encode_f32_map(fn, &tb, B, (uint64_t)K, (uint64_t)N, BN, BK, CU_TENSOR_MAP_SWIZZLE_NONE,
                        (uint64_t)tma.ldb))
        return cudaErrorInvalidValue;
    const bool c_vec = N % 4 == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0;
    auto kernel = c_vec ? sgemm_tma_streamk_kernel<true> : sgemm_tma_streamk_kernel<false>;
    static std::atomic<uint64_t> done_vec{0}, done_any{0};
    cudaError_t e = set_smem_limit_once(kernel, kSpreadSmem, c_vec ? done_vec : done_any);
    if (e != cudaSuccess)
        return e;
    // spread: reserve more than half of an SM's shared memory so that every
    // CTA has an SM to itself (the scheduler may otherwise pair CTAs on some
    // SMs and leave others idle).
    kernel<<<(unsigned)ctas, kThreads, spread ? kSpreadSmem : SMEM_BYTES, stream>>>(
        ta, tb, M, N, K, C, workspace, tma.err, tma.wait_limit_ns);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    // The fixup: a programmatic dependent of the stream-K grid, launched while
    // it runs and waiting for it inside the kernel.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, kFixupParts, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (c_vec)
        return cudaLaunchKernelEx(&cfg, sgemm_streamk_fixup_kernel<true>, (const float *)workspace, C,
                                  M, N, K, ctas);
    return cudaLaunchKernelEx(&cfg, sgemm_streamk_fixup_kernel<false>, (const float *)workspace, C,
                              M, N, K, ctas);
}

} // namespace rtm
