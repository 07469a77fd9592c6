// SIMT FP32 register-tiled product C = A.B for sm_103a.
//
// The three tiling levels of the register-tiling pages, re-sized for GB300:
//
//  * global tiling — each CTA owns one BM x BN tile of C; tiles are visited in
//    groups of GROUP_M tile-rows so CTAs resident together share A and B
//    panels in L2 ("寄存器Tiling跨架构解析", section 1.1: the global level fixes
//    block independence and global reuse);
//  * shared tiling — the CTA stages BK-deep K-slices of A and B in shared
//    memory through a STAGES-deep cp.async ring (zero-filled past M, N, K);
//    A is stored k-major (transposed) so a thread's column of A is one
//    128-bit load ("理解 Register Tiling", section "用一张图对比三个版本");
//  * register tiling — each of the 16 x 16 threads keeps a TM x TN fp32
//    accumulator tile and, for every k, loads TM values of A and TN values
//    of B into registers and forms their outer product with FFMA
//    ("理解 Register Tiling", section "关键循环：为什么省了 Shared Memory 读取？").
//
// GB300 choices that differ from the pages' 64x64-block / 4x4 example:
//  * 128 x 128 CTA tile, 8 x 8 per thread, split into 2 x 2 sub-blocks of
//    4 x 4 spaced 64 apart, so each thread's 8 A values and 8 B values are
//    two 128-bit shared loads each, and a warp's loads are conflict-free
//    (A: 4 distinct 16-byte granules per warp, B: 8 contiguous granules);
//  * per k: 64 FFMA per 4 LDS.128 (the pages' 4x4 tile gives 16 FFMA per
//    8 LDS.32); shared reads per output per k fall to (8+8)/64 = 0.25;
//  * the k-major A tile rows are padded by 4 floats (BM + 4 per k): a warp's
//    transposing 4-byte cp.async writes (4 rows x 8 k) then hit 32 distinct
//    banks, while reads stay 16-byte aligned and affine in k;
//  * __launch_bounds__(256, 2): at most 128 registers per thread, two CTAs
//    (16 warps) per SM; ptxas must report zero spill bytes.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace rtm {
namespace simt {

constexpr int kThreads = 256;  // 16 x 16 threads
constexpr int kGroupM = 8;     // tile-rows per L2 group

template <int BM, int BN, int BK, int STAGES>
struct Cfg {
    static constexpr int TM = BM / 16;
    static constexpr int TN = BN / 16;
    static constexpr int QM = TM / 4;       // 4x4 sub-blocks per thread along m
    static constexpr int QN = TN / 4;       // ... along n
    static constexpr int SUBM = BM / QM;    // distance between sub-blocks (64)
    static constexpr int SUBN = BN / QN;
    static constexpr int A_PER_THREAD = BM * BK / kThreads;        // 4-byte copies
    static constexpr int B4_PER_THREAD = BK * BN / 4 / kThreads;   // 16-byte copies
    static constexpr int B1_PER_THREAD = BK * BN / kThreads;       // 4-byte copies
    static constexpr int LDA = BM + 4;      // padded k-major A row
    static constexpr int SMEM_FLOATS = STAGES * BK * (LDA + BN);
    static constexpr size_t SMEM_BYTES = SMEM_FLOATS * sizeof(float);
    static_assert(TM % 4 == 0 && TN % 4 == 0, "thread tile is made of 4x4 sub-blocks");
    static_assert(BK % 8 == 0, "A loader covers k in groups of 8");
    static_assert(BM == 128 && BK % 8 == 0 && A_PER_THREAD == 4 * (BK / 8),
                  "A loader: warp w covers rows 16w..16w+15, 4 rows x 8 k per copy");
    static_assert(BK * BN % (4 * kThreads) == 0, "B loader coverage");
};

__device__ __forceinline__ void tile_of_block(int bid, int tiles_m, int tiles_n, int &tile_m,
                                              int &tile_n)
{
    const int group_size = kGroupM * tiles_n;
    const int group = bid / group_size;
    const int first_m = group * kGroupM;
    const int rows = min(tiles_m - first_m, kGroupM);
    const int in_group = bid - group * group_size;
    tile_m = first_m + in_group % rows;
    tile_n = in_group / rows;
}

template <int BM, int BN, int BK, int STAGES, bool B_VEC, bool C_VEC>
__global__ void __launch_bounds__(kThreads, 2)
    sgemm_rt_kernel(int M, int N, int K, const float *__restrict__ A,
                    const float *__restrict__ B, float *__restrict__ C)
{
    using G = Cfg<BM, BN, BK, STAGES>;
    constexpr int TM = G::TM, TN = G::TN, QM = G::QM, QN = G::QN;
    constexpr int SUBM = G::SUBM, SUBN = G::SUBN;

    constexpr int LDA = G::LDA;

    extern __shared__ __align__(16) float smem[];
    float *sA = smem;                           // [STAGES][BK][LDA], k-major A
    float *sB = smem + STAGES * BK * LDA;       // [STAGES][BK][BN]

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (N + BN - 1) / BN;
    int tile_m, tile_n;
    tile_of_block(blockIdx.x, tiles_m, tiles_n, tile_m, tile_n);
    const int m0 = tile_m * BM;
    const int n0 = tile_n * BN;

    // Thread (tm, tn) of the 16 x 16 grid; a warp is 4 (m) x 8 (n) threads.
    const int tm = (warp >> 1) * 4 + (lane >> 3);
    const int tn = (warp & 1) * 8 + (lane & 7);

    const int ktiles = (K + BK - 1) / BK;

    // A loader: copy (j, h) of this thread moves A[m0 + a_m + 4j][k0 + 8h + a_k]
    // (4-byte cp.async) to sA[8h + a_k][a_m + 4j]. A warp covers 4 rows x 8 k:
    // global reads are 32-byte runs, shared writes land in 32 distinct banks.
    const int a_m = warp * 16 + (lane >> 3);
    const int a_k = lane & 7;
    const float *a_src = A + (size_t)min(m0 + a_m, M - 1) * K + a_k;
    const size_t a_step4 = (size_t)4 * K;
    uint32_t a_rows_ok = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        a_rows_ok |= (m0 + a_m + 4 * j < M) ? (1u << j) : 0u;
    const uint32_t a_dst0 = smem_u32(sA + a_k * LDA + a_m);

    // B loader, 16-byte path: copy i moves B[k0 + 8i + warp][n0 + 4 lane .. +3]
    // (a warp reads one 512-byte row run). 4-byte path: copy i moves
    // B[k0 + 2i + tid / 128][n0 + tid % 128].
    const bool b_col_ok = B_VEC ? (n0 + lane * 4 < N) : true;

    auto load_tile = [&](int stage, int kt) {
        const int k0 = kt * BK;
        const uint32_t a_dst = a_dst0 + (uint32_t)(stage * BK * LDA) * 4u;
#pragma unroll
        for (int h = 0; h < BK / 8; ++h) {
            const bool k_ok = (k0 + 8 * h + a_k) < K;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool ok = k_ok && ((a_rows_ok >> j) & 1u);
                const float *src = ok ? a_src + a_step4 * j + (k0 + 8 * h) : A;
                cp_async_4(a_dst + (uint32_t)((8 * h * LDA + 4 * j) * 4), src, ok ? 4u : 0u);
            }
        }
        float *dB = sB + stage * BK * BN;
        if constexpr (B_VEC) {
#pragma unroll
            for (int i = 0; i < G::B4_PER_THREAD; ++i) {
                const int k = i * (kThreads / (BN / 4)) + tid / (BN / 4);
                const int n = (tid % (BN / 4)) * 4;
                const int gk = k0 + k;
                const bool ok = b_col_ok && (gk < K);  // N % 4 == 0: all four or none
                const float *src = ok ? B + (size_t)gk * N + (n0 + n) : B;
                cp_async_16(smem_u32(dB + k * BN + n), src, ok ? 16u : 0u);
            }
        } else {
#pragma unroll
            for (int i = 0; i < G::B1_PER_THREAD; ++i) {
                const int k = i * (kThreads / BN) + tid / BN;
                const int n = tid % BN;
                const int gk = k0 + k;
                const int gn = n0 + n;
                const bool ok = (gk < K) && (gn < N);
                const float *src = ok ? B + (size_t)gk * N + gn : B;
                cp_async_4(smem_u32(dB + k * BN + n), src, ok ? 4u : 0u);
            }
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j)
            acc[i][j] = 0.0f;

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < ktiles)
            load_tile(s, s);
        cp_async_commit();
    }

    for (int kt = 0; kt < ktiles; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();  // stage kt visible to all; stage kt-1 free for refill
        {
            const int nt = kt + STAGES - 1;
            if (nt < ktiles)
                load_tile(nt % STAGES, nt);
            cp_async_commit();
        }
        const int stage = kt % STAGES;
        const float *cA = sA + stage * BK * LDA + tm * 4;
        const float *cB = sB + stage * BK * BN + tn * 4;
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float a[TM], b[TN];
#pragma unroll
            for (int q = 0; q < QM; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(cA + k * LDA + q * SUBM);
                a[q * 4 + 0] = v.x;
                a[q * 4 + 1] = v.y;
                a[q * 4 + 2] = v.z;
                a[q * 4 + 3] = v.w;
            }
#pragma unroll
            for (int p = 0; p < QN; ++p) {
                const float4 v = *reinterpret_cast<const float4 *>(cB + k * BN + p * SUBN);
                b[p * 4 + 0] = v.x;
                b[p * 4 + 1] = v.y;
                b[p * 4 + 2] = v.z;
                b[p * 4 + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j)
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    cp_async_wait<0>();

    // Epilogue: masked stores, 128-bit where the row allows it.
#pragma unroll
    for (int q = 0; q < QM; ++q) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gm = m0 + q * SUBM + tm * 4 + i;
            if (gm >= M)
                continue;
            float *crow = C + (size_t)gm * N;
#pragma unroll
            for (int p = 0; p < QN; ++p) {
                const int gn = n0 + p * SUBN + tn * 4;
                const float *v = &acc[q * 4 + i][p * 4];
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

template <int BM, int BN, int BK, int STAGES, bool B_VEC, bool C_VEC>
cudaError_t launch_cfg(int M, int N, int K, const float *A, const float *B, float *C,
                       cudaStream_t stream)
{
    using G = Cfg<BM, BN, BK, STAGES>;
    auto kernel = sgemm_rt_kernel<BM, BN, BK, STAGES, B_VEC, C_VEC>;
    if (G::SMEM_BYTES > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)G::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
    }
    const long long tiles = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    if (tiles > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    kernel<<<(unsigned)tiles, kThreads, G::SMEM_BYTES, stream>>>(M, N, K, A, B, C);
    return cudaGetLastError();
}

} // namespace simt

cudaError_t launch_sgemm_f32(int M, int N, int K, const float *A, const float *B, float *C,
                             cudaStream_t stream)
{
    const bool b_vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(B) & 15) == 0);
    const bool c_vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15) == 0);
    constexpr int BM = 128, BN = 128, BK = 16, ST = 3;
    if (b_vec && c_vec)
        return simt::launch_cfg<BM, BN, BK, ST, true, true>(M, N, K, A, B, C, stream);
    if (b_vec)
        return simt::launch_cfg<BM, BN, BK, ST, true, false>(M, N, K, A, B, C, stream);
    if (c_vec)
        return simt::launch_cfg<BM, BN, BK, ST, false, true>(M, N, K, A, B, C, stream);
    return simt::launch_cfg<BM, BN, BK, ST, false, false>(M, N, K, A, B, C, stream);
}

} // namespace rtm
