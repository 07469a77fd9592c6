// The ablation ladder of the register-tiling page, on sm_103a: the kernels the
// page compares, kept as the page describes them so that their cost can be
// measured beside the tuned kernel ("【infra之路】理解 Register Tiling",
// sections "先看 Shared Memory 版本里，一个线程在做什么", "Register Tiling 的核心
// 思想", "关键循环：为什么省了 Shared Memory 读取？", "用一张图对比三个版本").
//
//   rung 0  naive: one thread per output, both operands read from global
//           memory (2K global reads per output);
//   rung 1  shared-memory tiled: 32 x 32 threads, TILE = 32, one output per
//           thread, sum += sA[ty][k] * sB[k][tx] (2 shared reads per output
//           per k);
//   rung 2  register tiled: 16 x 16 threads, 64 x 64 block, a 4 x 4 output
//           block per thread (rows ty*4.., columns tx*4..), regA[4] and regB[4]
//           loaded from shared memory per k, 16 FMA from registers (0.5 shared
//           reads per output per k); BK = 16.
//
// Rung 3 is the tuned kernel of sgemm_simt.cu (8 x 8 per thread, 0.25).
//
// Rungs 4-6 are the page's extreme-tile experiment ("寄存器Tiling跨架构解析",
// section 7.4: time the kernel with a 1x1 and with a large tile to see how much
// register tiling contributes): rung 2's kernel, unchanged but for the size of
// the per-thread tile T x T, on the same 16 x 16 threads and BK = 16, so the
// block is 16T x 16T and a thread reads 2T values from shared memory for T^2
// FMA (2/T shared reads per output per k):
//   rung 4  T = 1 (16 x 16 block, 2 reads per output per k);
//   rung 5  T = 2 (32 x 32 block, 1);
//   rung 2  T = 4 (64 x 64 block, 0.5);
//   rung 6  T = 8 (128 x 128 block, 0.25).
// All rungs handle ragged M, N, K: out-of-range loads read zeros, stores are
// masked.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"

namespace rtm {
namespace ladder {

__global__ void naive_kernel(int M, int N, int K, const float *__restrict__ A,
                             const float *__restrict__ B, float *__restrict__ C)
{
    const int row = blockIdx.y * 16 + threadIdx.y;
    const int col = blockIdx.x * 16 + threadIdx.x;
    if (row >= M || col >= N)
        return;
    float sum = 0.0f;
    for (int k = 0; k < K; ++k)
        sum += A[(size_t)row * K + k] * B[(size_t)k * N + col];
    C[(size_t)row * N + col] = sum;
}

constexpr int TILE = 32;

__global__ void __launch_bounds__(TILE *TILE)
    shared_tiled_kernel(int M, int N, int K, const float *__restrict__ A,
                        const float *__restrict__ B, float *__restrict__ C)
{
    __shared__ float sA[TILE][TILE];
    __shared__ float sB[TILE][TILE];
    const int ty = threadIdx.y, tx = threadIdx.x;
    const int row = blockIdx.y * TILE + ty;
    const int col = blockIdx.x * TILE + tx;
    float sum = 0.0f;
    for (int k0 = 0; k0 < K; k0 += TILE) {
        sA[ty][tx] = (row < M && k0 + tx < K) ? A[(size_t)row * K + k0 + tx] : 0.0f;
        sB[ty][tx] = (k0 + ty < K && col < N) ? B[(size_t)(k0 + ty) * N + col] : 0.0f;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < TILE; ++k)
            sum += sA[ty][k] * sB[k][tx];
        __syncthreads();
    }
    if (row < M && col < N)
        C[(size_t)row * N + col] = sum;
}

constexpr int RT = 16;       // threads per side
constexpr int BK = 16;

// T x T outputs per thread (the page's kernel has T = 4: a 64 x 64 block).
template <int T>
__global__ void __launch_bounds__(RT *RT)
    register_tiled_kernel(int M, int N, int K, const float *__restrict__ A,
                          const float *__restrict__ B, float *__restrict__ C)
{
    constexpr int TM = T, TN = T;
    constexpr int BM = RT * TM;
    constexpr int BN = RT * TN;
    __shared__ float sA[BM][BK];
    __shared__ float sB[BK][BN];
    const int ty = threadIdx.y, tx = threadIdx.x;
    const int tid = ty * RT + tx;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int thread_row = ty * TM, thread_col = tx * TN;

    float results[TM][TN] = {};
    for (int k0 = 0; k0 < K; k0 += BK) {
        // cooperative load: BM x BK of A and BK x BN of B, 4 elements each
#pragma unroll
        for (int i = 0; i < BM * BK / (RT * RT); ++i) {
            const int e = i * RT * RT + tid;
            const int r = e / BK, kk = e % BK;
            sA[r][kk] = (m0 + r < M && k0 + kk < K) ? A[(size_t)(m0 + r) * K + k0 + kk] : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < BK * BN / (RT * RT); ++i) {
            const int e = i * RT * RT + tid;
            const int kk = e / BN, c = e % BN;
            sB[kk][c] = (k0 + kk < K && n0 + c < N) ? B[(size_t)(k0 + kk) * N + n0 + c] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float regA[TM], regB[TN];
#pragma unroll
            for (int m = 0; m < TM; ++m)
                regA[m] = sA[thread_row + m][k];
#pragma unroll
            for (int n = 0; n < TN; ++n)
                regB[n] = sB[k][thread_col + n];
#pragma unroll
            for (int m = 0; m < TM; ++m)
#pragma unroll
                for (int n = 0; n < TN; ++n)
                    results[m][n] += regA[m] * regB[n];
        }
        __syncthreads();
    }
#pragma unroll
    for (int m = 0; m < TM; ++m) {
        const int r = m0 + thread_row + m;
        if (r >= M)
            continue;
#pragma unroll
        for (int n = 0; n < TN; ++n) {
            const int c = n0 + thread_col + n;
            if (c < N)
                C[(size_t)r * N + c] = results[m][n];
        }
    }
}

} // namespace ladder

cudaError_t launch_sgemm_ladder(int rung, int M, int N, int K, const float *A, const float *B,
                                float *C, cudaStream_t stream)
{
    using namespace ladder;
    // Grids are (N / tile) x (M / tile); the y extent is limited to 65535.
    static const int kTile[7] = {16, TILE, RT * 4, 0, RT * 1, RT * 2, RT * 8};
    if (rung < 0 || rung > 6 || rung == 3)
        return cudaErrorInvalidValue;
    const int tile = kTile[rung];
    if ((M + tile - 1) / tile > 65535)
        return cudaErrorInvalidValue;
    switch (rung) {
    case 0: {
        dim3 grid((N + 15) / 16, (M + 15) / 16);
        naive_kernel<<<grid, dim3(16, 16), 0, stream>>>(M, N, K, A, B, C);
        break;
    }
    case 1: {
        dim3 grid((N + TILE - 1) / TILE, (M + TILE - 1) / TILE);
        shared_tiled_kernel<<<grid, dim3(TILE, TILE), 0, stream>>>(M, N, K, A, B, C);
        break;
    }
    case 2:
    case 4:
    case 5:
    case 6: {
        dim3 grid((N + tile - 1) / tile, (M + tile - 1) / tile);
        if (rung == 2)
            register_tiled_kernel<4><<<grid, dim3(RT, RT), 0, stream>>>(M, N, K, A, B, C);
        else if (rung == 4)
            register_tiled_kernel<1><<<grid, dim3(RT, RT), 0, stream>>>(M, N, K, A, B, C);
        else if (rung == 5)
            register_tiled_kernel<2><<<grid, dim3(RT, RT), 0, stream>>>(M, N, K, A, B, C);
        else
            register_tiled_kernel<8><<<grid, dim3(RT, RT), 0, stream>>>(M, N, K, A, B, C);
        break;
    }
    default:
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

} // namespace rtm
