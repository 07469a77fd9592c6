// SIMT FP32 product C = A.B for short, wide products (M <= 32) on sm_103a.
//
// With few rows of A the 128 x 128 tiles of sgemm_simt.cu compute mostly
// rows of zeros (M = 16 leaves 7/8 of every tile empty), and the product is
// bound by reading B once from HBM. Here the register tile is a column strip
// ("理解 Register Tiling", section "Register Tiling 的核心思想": a thread keeps a
// TM x TN block of outputs in registers and reuses every loaded value across
// it; here TN = 2 and TM = MR >= M):
//
//  * global tiling — a CTA owns 256 columns of C and, when that leaves SMs
//    idle, one of S K-ranges (S = 2, 4 or 8 CTAs of one cluster split K);
//  * shared tiling — a 6-stage cp.async ring of 16-deep K-slices (about
//    100 KB of B in flight per CTA, two CTAs per SM: on GB300 one SM streams
//    only 30-40 GB/s with 100-160 KB outstanding, so reading B at HBM speed
//    takes most SMs, and two rings per SM let K be split eight ways with
//    every cluster resident; 10 stages at one CTA per SM were 16-26 % slower:
//    1 x 8192 x 8192 61.5 -> 51.7 us, 16 x 8192 x 8192 108.6 -> 82.0 us):
//    B as stored (16 x 256, 16-byte copies where B's rows allow) and A
//    transposed to k-major (16 x MR, rows padded to MR + 4 floats);
//  * register tiling — thread t keeps C[0..MR)[n0 + 2t .. n0 + 2t + 1] in
//    registers; per k it reads two B values (one 64-bit read; consecutive
//    threads, consecutive words) and MR values of A (128-bit broadcast reads)
//    and issues 2 MR FMA, so each B value is used MR times and each A value
//    twice;
//  * epilogue — with S = 1 each thread stores its two columns (for each row
//    the 128 threads write 256 consecutive floats). With S > 1 each CTA writes
//    its MR x 256 partial into its idle stage memory; after a cluster barrier CTA
//    r sums rows [r MR / S, (r+1) MR / S) over the S partials, read through
//    distributed shared memory in rank order (the same sum on every call),
//    and a second cluster barrier keeps every partial alive until all have
//    been read.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace rtm {
namespace sshort {

constexpr int BN = 256;      // columns of C per CTA
constexpr int BK = 16;       // K-slice depth
constexpr int STAGES = 6;    // about 100 KB of B in flight per CTA, two CTAs per SM

template <int MR>
struct Cfg {
    static constexpr int APITCH = MR + 4;  // floats per k-row of the A slice
    static constexpr int B_FLOATS = BK * BN;
    static constexpr int A_FLOATS = BK * APITCH;
    static constexpr int STAGE_FLOATS = B_FLOATS + A_FLOATS;
    static constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_FLOATS * 4;
    static_assert(MR * BN <= STAGES * STAGE_FLOATS, "partial sums must fit the stage ring");
};

// TN columns of C per thread (BN / TN threads per CTA).
template <int MR, int TN, bool B_VEC>
__global__ void __launch_bounds__(BN / TN, 1)
    sgemm_short_kernel(int M, int N, int K, const float *__restrict__ A,
                       const float *__restrict__ B, float *__restrict__ C, int splits)
{
    constexpr int kThreads = BN / TN;
    using G = Cfg<MR>;
    extern __shared__ __align__(16) float smem[];
    const int t = threadIdx.x;
    const int S = splits;
    const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
    const int n0 = (blockIdx.x / S) * BN;
    // This CTA's K-range, a whole number of slices.
    const int slices = (K + BK - 1) / BK;
    const int per = (slices + S - 1) / S;
    const int s_begin = min(slices, (int)rank * per);
    const int s_end = min(slices, s_begin + per);
    const int nslices = s_end - s_begin;

    auto stage_b = [&](int s) { return smem + s * G::STAGE_FLOATS; };
    auto stage_a = [&](int s) { return smem + s * G::STAGE_FLOATS + G::B_FLOATS; };

    // Copies of one slice into stage s; zeros outside M, N and K.
    auto load = [&](int slice, int s) {
        const int k0 = (s_begin + slice) * BK;
        float *sb = stage_b(s);
        if constexpr (B_VEC) {
            const int c4 = (t % (BN / 4)) * 4;  // 64 chunks of 4 floats per row
#pragma unroll
            for (int j = 0; j < BK * BN / 4 / kThreads; ++j) {
                const int kk = t / (BN / 4) + j * (kThreads / (BN / 4));
                const int gk = k0 + kk, gn = n0 + c4;
                const bool in = gk < K && gn < N;
                cp_async_16(smem_u32(sb + kk * BN + c4), in ? B + (size_t)gk * N + gn : B,
                            in ? 16u : 0u);
            }
        } else {
#pragma unroll 4
            for (int kk = 0; kk < BK; ++kk) {
#pragma unroll
                for (int c = 0; c < TN; ++c) {
                    const int col = TN * t + c;
                    const int gk = k0 + kk, gn = n0 + col;
                    const bool in = gk < K && gn < N;
                    cp_async_4(smem_u32(sb + kk * BN + col), in ? B + (size_t)gk * N + gn : B,
                               in ? 4u : 0u);
                }
            }
        }
        // A: MR x 16 values, read along k (coalesced), stored k-major.
        float *sa = stage_a(s);
        for (int e = t; e < MR * BK; e += kThreads) {
            const int kk = e % BK, m = e / BK;
            const int gk = k0 + kk;
            const bool in = m < M && gk < K;
            cp_async_4(smem_u32(sa + kk * G::APITCH + m), in ? A + (size_t)m * K + gk : A,
                       in ? 4u : 0u);
        }
    };

    float acc[MR][TN];
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
        for (int c = 0; c < TN; ++c)
            acc[m][c] = 0.0f;

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < nslices)
            load(s, s);
        cp_async_commit();
    }
    for (int i = 0; i < nslices; ++i) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        const int s = i % STAGES;
        const float *sb = stage_b(s);
        const float *sa = stage_a(s);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float b[TN];
            if constexpr (TN == 2) {
                const float2 b2 = *reinterpret_cast<const float2 *>(sb + kk * BN + TN * t);
                b[0] = b2.x;
                b[TN - 1] = b2.y;
            } else {
                b[0] = sb[kk * BN + t];
            }
#pragma unroll
            for (int q = 0; q < MR / 4; ++q) {
                const float4 a = *reinterpret_cast<const float4 *>(sa + kk * G::APITCH + 4 * q);
#pragma unroll
                for (int c = 0; c < TN; ++c) {
                    acc[4 * q + 0][c] = fmaf(a.x, b[c], acc[4 * q + 0][c]);
                    acc[4 * q + 1][c] = fmaf(a.y, b[c], acc[4 * q + 1][c]);
                    acc[4 * q + 2][c] = fmaf(a.z, b[c], acc[4 * q + 2][c]);
                    acc[4 * q + 3][c] = fmaf(a.w, b[c], acc[4 * q + 3][c]);
                }
            }
        }
        // Refill the stage that was consumed one iteration ago.
        const int next = i + STAGES - 1;
        if (next < nslices)
            load(next, next % STAGES);
        cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();

    const int gn = n0 + TN * t;
    if (S == 1) {
#pragma unroll
        for (int m = 0; m < MR; ++m)
            if (m < M) {
                float *cp = C + (size_t)m * N + gn;
#pragma unroll
                for (int c = 0; c < TN; ++c)
                    if (gn + c < N)
                        cp[c] = acc[m][c];
            }
        return;
    }
    // Partial sums, row m of the partial at smem[m * BN + col].
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
        for (int c = 0; c < TN; ++c)
            smem[m * BN + TN * t + c] = acc[m][c];
    cluster_sync();
    const int rows = MR / S;
    const int r0 = (int)rank * rows;
    for (int m = r0; m < r0 + rows; ++m) {
#pragma unroll
        for (int c = 0; c < TN; ++c) {
            const uint32_t mine = smem_u32(smem + m * BN + TN * t + c);
            float sum = ld_shared_cluster_f32(mapa_shared(mine, 0));
            for (int q = 1; q < S; ++q)
                sum += ld_shared_cluster_f32(mapa_shared(mine, (uint32_t)q));
            if (m < M && gn + c < N)
                C[(size_t)m * N + gn + c] = sum;
        }
    }
    cluster_sync();
}

template <int MR, int TN, bool B_VEC>
static cudaError_t launch(int M, int N, int K, const float *A, const float *B, float *C,
                          int splits, cudaStream_t stream)
{
    auto kernel = sgemm_short_kernel<MR, TN, B_VEC>;
    static std::atomic<uint64_t> done{0};
    cudaError_t e = set_smem_limit_once(kernel, (int)Cfg<MR>::SMEM_BYTES, done);
    if (e != cudaSuccess)
        return e;
    const long long blocks = (long long)((N + BN - 1) / BN) * splits;
    if (blocks > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(BN / TN, 1, 1);
    cfg.dynamicSmemBytes = Cfg<MR>::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, M, N, K, A, B, C, splits);
}

template <int MR, int TN>
static cudaError_t launch_b(int M, int N, int K, const float *A, const float *B, float *C,
                            int splits, cudaStream_t stream)
{
    const bool b_vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(B) & 15) == 0);
    return b_vec ? launch<MR, TN, true>(M, N, K, A, B, C, splits, stream)
                 : launch<MR, TN, false>(M, N, K, A, B, C, splits, stream);
}

} // namespace sshort

// How many clusters of 8 CTAs of this kernel can be resident at once on the
// current device (cached; 0 if unknown).
static int resident_clusters_of_8()
{
    auto kernel = sshort::sgemm_short_kernel<32, 2, true>;
    static std::atomic<uint64_t> done{0};
    if (set_smem_limit_once(kernel, (int)sshort::Cfg<32>::SMEM_BYTES, done) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    static std::atomic<int> cache[64] = {};
    return resident_clusters(kernel, 8, sshort::BN / 2, sshort::Cfg<32>::SMEM_BYTES, cache);
}

int sgemm_short_splits(int M, int N, int K, int sm_count)
{
    (void)M;
    const long long blocks = (N + sshort::BN - 1) / sshort::BN;
    int splits = 1;
    // Up to two CTAs per SM, at least 256 of K per CTA.
    while (splits < 8 && blocks * splits * 2 <= 2LL * sm_count && K / (splits * 2) >= 256)
        splits *= 2;
    // A cluster that must wait for another to finish doubles the time, so 8
    // only when every cluster of 8 is resident at once.
    if (splits == 8 && blocks > resident_clusters_of_8())
        splits = 4;
    return splits;
}

cudaError_t launch_sgemm_short(int M, int N, int K, const float *A, const float *B, float *C,
                               int splits, cudaStream_t stream)
{
    using namespace sshort;
    if (M < 1 || M > kShortMaxM || (splits != 1 && splits != 2 && splits != 4 && splits != 8))
        return cudaErrorInvalidValue;
    // Two columns per thread (128 threads): measured faster than one column per
    // thread (256 threads) on every shape tried, e.g. 32 x 8192 x 8192 0.168 ms
    // against 0.205 ms.
    if (M <= 8)
        return launch_b<8, 2>(M, N, K, A, B, C, splits, stream);
    if (M <= 16)
        return launch_b<16, 2>(M, N, K, A, B, C, splits, stream);
    return launch_b<32, 2>(M, N, K, A, B, C, splits, stream);
}

} // namespace rtm
