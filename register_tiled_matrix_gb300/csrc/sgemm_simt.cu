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
//    CTAs whose tile lies inside M x N copy full slices without predicates,
//    interleaved with the FFMA of the current slice over its first 5/8;
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
//  * the 64 FFMA of a k-step walk the 8 x 8 accumulator tile in serpentine
//    order (odd rows backwards), so consecutive FFMA always share an operand
//    and the hardware operand-reuse cache can serve it (measured: +4 % over
//    row-by-row order on GB300);
//  * products with N <= 64 use 128 x 64 tiles (8 x 4 per thread), or
//    256 x 64 (16 x 4) where the schedule model prices them lower;
//  * BK = 32 with two stages (66.6 KB of shared memory per CTA): a sweep of
//    BK in {8..48} and 2-4 stages on GB300 put this on top (59 TFLOP/s at
//    4096^3 against 56 for three stages);
//  * __launch_bounds__(256, 2): at most 128 registers per thread, two CTAs
//    (16 warps) per SM; ptxas must report zero spill bytes.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace rtm {
namespace simt {

constexpr int kThreads = 256;  // 16 x 16 threads
// Tile-rows per L2 group: the TMA-fed kernels' value, so that both visit the
// tiles in the same order and a ragged last wave split over clusters holds
// the same tiles whichever kernel stages the operands (the same bits).
constexpr int kGroupM = 16;

// How K is split (one CTA per K chunk and C tile; the chunk index is blockIdx.y).
enum SplitMode : int {
    kPlain = 0,           // no split: gridDim.y == 1
    kSplitWorkspace = 1,  // each chunk writes its partial tile to its own slab of a workspace
    kSplitCluster = 2,    // the chunks of one tile are one cluster and add their partial
                          // tiles through distributed shared memory
};

template <int BM, int BN, int BK, int STAGES>
struct Cfg {
    static constexpr int JROWS = BM / 32;   // A copies per thread per 8-deep k group
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
    static_assert(BM % 32 == 0 && A_PER_THREAD == JROWS * (BK / 8),
                  "A loader: warp w covers rows w*BM/8 .. +BM/8, 4 rows x 8 k per copy");
    static_assert(BK * BN % (4 * kThreads) == 0, "B loader coverage");
    static constexpr int FAST_COPIES = A_PER_THREAD + B4_PER_THREAD;
    // kSplitCluster: the partial tile parked in shared memory after the k loop,
    // rows padded by 4 floats (a quarter-warp's 128-bit stores, 2 rows 4 apart
    // x 64 bytes, then fall in distinct banks).
    static constexpr int PART_PITCH = BN + 4;
    static constexpr size_t PART_BYTES = (size_t)BM * PART_PITCH * sizeof(float);
    static constexpr size_t CLUSTER_SMEM_BYTES = SMEM_BYTES > PART_BYTES ? SMEM_BYTES : PART_BYTES;
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

// kSplitCluster, after the cluster barrier: CTA r of the S = gridDim.y CTAs of
// a cluster adds rows [r * BM / S, +BM / S) of the S partial tiles parked in
// the cluster's shared memory (row pitch PITCH), reading them through
// distributed shared memory in rank order, and stores the sums to C with the
// same masks as the plain epilogue. S is a template constant so that every
// load of a thread is issued before its first add and the distributed-shared-
// memory latency is paid about once (2048 x 640 x 2048, clusters of 8, on
// GB300: 133.8 -> 124.3 us). Kept out of line: inlined, it cost the k loop of
// the 4-byte-copy variant spilled registers.
template <int BM, int BN, int PITCH, bool C_VEC, int S>
__device__ __noinline__ void cluster_add_partials(const float *part, int M, int N, float *C,
                                                  int first_tile)
{
    int tile_m, tile_n;
    tile_of_block((int)blockIdx.x + first_tile, (M + BM - 1) / BM, (N + BN - 1) / BN, tile_m,
                  tile_n);
    // The partial tiles start at the k loop's (possibly shifted) tile origin;
    // only the tile's own rows and columns, from m0s and n0s on, are stored.
    const int m0s = tile_m * BM, n0s = tile_n * BN;
    const bool shift = M >= BM && N >= BN;
    const int m0 = shift ? min(m0s, M - BM) : m0s;
    const int n0 = shift ? min(n0s, N - BN) : n0s;
    const int rank = (int)blockIdx.y;  // cluster of (1, S, 1)
    constexpr int ROWS = BM / S;
    constexpr int COUNT4 = ROWS * (BN / 4);
    constexpr int ITERS = (COUNT4 + kThreads - 1) / kThreads;
    float4 v[ITERS][S];  // at most 16 float4 for every tile shape and S
#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
        const int f = (int)threadIdx.x + it * kThreads;
        if (COUNT4 % kThreads == 0 || f < COUNT4) {
            const int r = rank * ROWS + f / (BN / 4);
            const int c = (f % (BN / 4)) * 4;
            const uint32_t local = smem_u32(part + r * PITCH + c);
#pragma unroll
            for (int q = 0; q < S; ++q)
                v[it][q] = ld_shared_cluster_v4(mapa_shared(local, (uint32_t)q));
        }
    }
#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
        const int f = (int)threadIdx.x + it * kThreads;
        if (!(COUNT4 % kThreads == 0 || f < COUNT4))
            continue;
        float4 sum = v[it][0];
#pragma unroll
        for (int q = 1; q < S; ++q) {
            sum.x += v[it][q].x;
            sum.y += v[it][q].y;
            sum.z += v[it][q].z;
            sum.w += v[it][q].w;
        }
        const int r = rank * ROWS + f / (BN / 4);
        const int c = (f % (BN / 4)) * 4;
        const int gm = m0 + r, gn = n0 + c;
        if (gm < M && gm >= m0s) {
            float *crow = C + (size_t)gm * N;
            if constexpr (C_VEC) {
                if (gn < N && gn >= n0s)
                    *reinterpret_cast<float4 *>(crow + gn) = sum;
            } else {
                const float w[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (gn + j < N && gn + j >= n0s)
                        crow[gn + j] = w[j];
            }
        }
    }
}

// ORDER 0: accumulator tile walked row by row; 1: serpentine (odd rows walk
// the columns backwards, so the B operand of a row's last FFMA is the first of
// the next row's and can be reused by the operand cache).
template <int BM, int BN, int BK, int STAGES, int MINB, int ORDER, bool B_VEC, bool C_VEC,
          int SPLIT>
__global__ void __launch_bounds__(kThreads, MINB)
    sgemm_rt_kernel(int M, int N, int K_total, int kchunk, const float *__restrict__ A,
                    const float *__restrict__ B, float *__restrict__ C, size_t aux)
{
    // Split-K: CTA row blockIdx.y of the grid sums k in [y * kchunk, +kchunk);
    // A keeps its full row stride K_total. kSplitWorkspace writes the partial
    // tile to C + y * aux (aux: floats between slabs); kSplitCluster adds the
    // partial tiles of the cluster's CTAs (the K chunks of one tile) after the
    // k loop, and its grid covers tiles aux .. aux + gridDim.x - 1 (a plain
    // grid always starts at tile 0 and may stop early). The plain
    // product is compiled without any of this (the extra runtime offsets changed
    // the register allocation of the FFMA loop and cost 6 % on GB300).
    int lda = K_total;
    int K = K_total;
    if constexpr (SPLIT != kPlain) {
        const int k_begin = blockIdx.y * kchunk;
        K = min(kchunk, K_total - k_begin);
        A += k_begin;
        B += (size_t)k_begin * N;
        if constexpr (SPLIT == kSplitWorkspace) {
            C += blockIdx.y * aux;
            grid_launch_dependents();  // the reduction may launch; it waits for this grid
        }
    }

    using G = Cfg<BM, BN, BK, STAGES>;
    constexpr int TM = G::TM, TN = G::TN, QM = G::QM, QN = G::QN;
    constexpr int SUBM = G::SUBM, SUBN = G::SUBN;
    constexpr int LDA = G::LDA;
    constexpr uint32_t A_STAGE_BYTES = BK * LDA * 4;
    constexpr uint32_t B_STAGE_BYTES = BK * BN * 4;

    extern __shared__ __align__(16) float smem[];
    float *sA = smem;                           // [STAGES][BK][LDA], k-major A
    float *sB = smem + STAGES * BK * LDA;       // [STAGES][BK][BN]

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (N + BN - 1) / BN;
    int tile_m, tile_n;
    if constexpr (SPLIT == kSplitCluster)
        tile_of_block((int)blockIdx.x + (int)aux, tiles_m, tiles_n, tile_m, tile_n);
    else
        tile_of_block(blockIdx.x, tiles_m, tiles_n, tile_m, tile_n);
    // kSplitCluster: edge tiles of a product at least one tile high and wide
    // compute the last BM x BN block of C instead, shifted back over their
    // neighbours, so that every full K-slice is copied without predicates;
    // they store only their own rows and columns (from m0s, n0s on). On GB300:
    // 1000 x 1000 x 999 split 4 57.5 -> 53.4 us, 300 x 201 x 1024 split 8
    // 22.7 -> 20.6 us. The plain product keeps predicated edge tiles: the same
    // change there cost the FFMA loop's register allocation 8 % at 4096^3.
    const int m0s = tile_m * BM, n0s = tile_n * BN;
    const bool shift = SPLIT == kSplitCluster && M >= BM && N >= BN;
    const int m0 = shift ? min(m0s, M - BM) : m0s;
    const int n0 = shift ? min(n0s, N - BN) : n0s;

    // Thread (tm, tn) of the 16 x 16 grid; a warp is 4 (m) x 8 (n) threads
    // and each quarter-warp 2 (m) x 4 (n), so that every 128-bit fragment
    // load of a half-warp needs one shared-memory wavefront (broadcast merges
    // only inside a quarter-warp).
    const int tm = (warp >> 1) * 4 + (((lane >> 2) & 1) | ((lane >> 3) & 2));
    const int tn = (warp & 1) * 8 + ((lane & 3) | ((lane >> 1) & 4));

    const int ktiles = (K + BK - 1) / BK;
    // K-slices that lie wholly inside K; with the tile wholly inside M x N
    // they are loaded without any predicate.
    const bool interior = (m0 + BM <= M) && (n0 + BN <= N);
    const int kfull = interior ? K / BK : 0;

    // A loader: copy (j, h) of this thread moves A[m0 + a_m + 4j][k0 + 8h + a_k]
    // (4-byte cp.async) to sA[8h + a_k][a_m + 4j]. A warp covers 4 rows x 8 k:
    // global reads are 32-byte runs, shared writes land in 32 distinct banks.
    constexpr int JROWS = G::JROWS;
    const int a_m = warp * (BM / 8) + (lane >> 3);
    const int a_k = lane & 7;
    const float *a_src = A + (size_t)min(m0 + a_m, M - 1) * lda + a_k;
    const uint32_t a_dst0 = smem_u32(sA + a_k * LDA + a_m);

    // B loader, 16-byte path: copy i moves B[k0 + 8i + warp][n0 + 4 lane .. +3]
    // (a warp reads one 512-byte row run). 4-byte path: copy i moves
    // B[k0 + 2i + tid / 128][n0 + tid % 128].
    // (BN = 128: a warp moves one 512-byte row; narrower tiles: BN / 4 threads
    // per row.)
    uint32_t b_dst0;
    if constexpr (BN == 128)
        b_dst0 = smem_u32(sB + warp * BN + lane * 4);
    else
        b_dst0 = smem_u32(sB + (tid / (BN / 4)) * BN + (tid % (BN / 4)) * 4);

    // 4-byte B path: this thread's column and first row of every slice.
    const float *b1_src = B + (size_t)(tid / BN) * N + (n0 + tid % BN);
    const uint32_t b1_dst0 = smem_u32(sB + (tid / BN) * BN + tid % BN);
    const float *b1_next = b1_src;

    // Unpredicated copies of K-slice kt into `stage` (interior tiles, full
    // slices), one per call so they can be spread over the FMA loop: copies
    // 0 .. A_PER_THREAD-1 are A elements, the rest B vectors (16-byte path) or
    // B elements (4-byte path, rows of B not on 16-byte boundaries).
    constexpr int FAST_COPIES =
        B_VEC ? G::FAST_COPIES : G::A_PER_THREAD + G::B1_PER_THREAD;
    // The copies are spread over the first 5/8 of the k loop, so that the
    // last of them still has a few k-steps to land before the wait at the top
    // of the next iteration: one per k for the 20 copies of the 16-byte path,
    // two per k for the 32 of the 4-byte path (one per k there left the last
    // copy issued just before that wait; 2 % slower at 4096 x 4093 x 4096 on
    // GB300). The cluster-split 4-byte variant keeps one per k: two cost it a
    // 16-byte register spill.
    constexpr int COPY_SPAN = (SPLIT == kSplitCluster && !B_VEC) ? BK : BK * 5 / 8;
    constexpr int COPIES_PER_K = (FAST_COPIES + COPY_SPAN - 1) / COPY_SPAN;
    auto fast_copy = [&](int c, uint32_t stage, int kt) {
        const int k0 = kt * BK;
        if (c < G::A_PER_THREAD) {
            const int h = c / JROWS, j = c % JROWS;
            cp_async_4_full(a_dst0 + stage * A_STAGE_BYTES + (uint32_t)((8 * h * LDA + 4 * j) * 4),
                            a_src + (size_t)(4 * j) * lda + (k0 + 8 * h));
        } else if constexpr (!B_VEC) {
            // copy i moves B[k0 + i * (256 / BN) + tid / BN][n0 + tid % BN]. The
            // source walks down B from the slice's first row, one pointer bump
            // per copy: with a separate offset per copy the compiler kept the
            // 16 offsets live across the loop, and the FFMA loop's register
            // allocation suffered (4096 x 4093 x 4096 on GB300: 2.655 -> 2.527
            // ms; the same chain for the A copies slowed 4096^3 by 6 %).
            // The cluster-split variant keeps the per-copy offsets: with the
            // chain it spilled 32 bytes.
            const int i = c - G::A_PER_THREAD;
            if constexpr (SPLIT == kSplitCluster) {
                const int k = i * (kThreads / BN) + tid / BN;
                const int n = tid % BN;
                cp_async_4_full(smem_u32(sB + stage * (BK * BN) + k * BN + n),
                                B + (size_t)(k0 + k) * N + (n0 + n));
            } else {
                if (i == 0)
                    b1_next = b1_src + (size_t)k0 * N;
                cp_async_4_full(b1_dst0 + stage * B_STAGE_BYTES +
                                    (uint32_t)(i * (kThreads / BN) * BN * 4),
                                b1_next);
                b1_next += (size_t)(kThreads / BN) * N;
            }
        } else {
            const int i = c - G::A_PER_THREAD;
            const int krow = i * (kThreads / (BN / 4));
            if constexpr (BN == 128)
                cp_async_16_full(b_dst0 + stage * B_STAGE_BYTES + (uint32_t)(krow * BN * 4),
                                 B + (size_t)(k0 + krow + warp) * N + (n0 + lane * 4));
            else
                cp_async_16_full(b_dst0 + stage * B_STAGE_BYTES + (uint32_t)(krow * BN * 4),
                                 B + (size_t)(k0 + krow + tid / (BN / 4)) * N +
                                     (n0 + (tid % (BN / 4)) * 4));
        }
    };

    // Predicated copy: zero-fills everything outside M, N, K.
    auto load_pred = [&](uint32_t stage, int kt) {
        const int k0 = kt * BK;
        const uint32_t a_dst = a_dst0 + stage * A_STAGE_BYTES;
#pragma unroll
        for (int h = 0; h < BK / 8; ++h) {
            const bool k_ok = (k0 + 8 * h + a_k) < K;
#pragma unroll
            for (int j = 0; j < JROWS; ++j) {
                const bool ok = k_ok && (m0 + a_m + 4 * j < M);
                const float *src = ok ? a_src + (size_t)(4 * j) * lda + (k0 + 8 * h) : A;
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
                const bool ok = (n0 + n < N) && (gk < K);  // N % 4 == 0: all four or none
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

    auto load_tile = [&](uint32_t stage, int kt) {
        if (kt < kfull) {
#pragma unroll
            for (int c = 0; c < FAST_COPIES; ++c)
                fast_copy(c, stage, kt);
        } else {
            load_pred(stage, kt);
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

    uint32_t read_stage = 0;
    uint32_t write_stage = STAGES - 1;
    for (int kt = 0; kt < ktiles; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();  // slice kt visible to all; the stage read at kt-1 is free
        const int nt = kt + STAGES - 1;
        const bool fast = nt < kfull;  // copies spread over the FMA loop below
        if (!fast && nt < ktiles)
            load_pred(write_stage, nt);
        const uint32_t fill_stage = write_stage;
        write_stage = (write_stage + 1 == STAGES) ? 0 : write_stage + 1;
        const float *cA = sA + read_stage * (BK * LDA) + tm * 4;
        const float *cB = sB + read_stage * (BK * BN) + tn * 4;
        read_stage = (read_stage + 1 == STAGES) ? 0 : read_stage + 1;
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
                for (int jj = 0; jj < TN; ++jj) {
                    const int j = (ORDER == 1 && (i & 1)) ? TN - 1 - jj : jj;
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                }
#pragma unroll
            for (int q = 0; q < COPIES_PER_K; ++q)
                if (fast && k * COPIES_PER_K + q < FAST_COPIES)
                    fast_copy(k * COPIES_PER_K + q, fill_stage, nt);
        }
        cp_async_commit();
    }
    cp_async_wait<0>();

    if constexpr (SPLIT == kSplitCluster) {
        // Every CTA parks its partial tile in its own (now idle) shared memory;
        // after a cluster barrier CTA r adds rows [r * BM / S, +BM / S) of the S
        // partial tiles, read through distributed shared memory in rank order
        // (so the sum is the same on every call), and stores them. The second
        // barrier keeps each CTA's partial alive until every CTA has read it.
        constexpr int PITCH = G::PART_PITCH;
        // The thread and tile coordinates are read again from the special
        // registers rather than kept live across the k loop, where the
        // 128-register budget has no room for them.
        const int tid2 = (int)special_tid_x();
        const int warp2 = tid2 >> 5, lane2 = tid2 & 31;
        const int tm2 = (warp2 >> 1) * 4 + (((lane2 >> 2) & 1) | ((lane2 >> 3) & 2));
        const int tn2 = (warp2 & 1) * 8 + ((lane2 & 3) | ((lane2 >> 1) & 4));
        __syncthreads();  // every warp has finished reading the last K-slice
#pragma unroll
        for (int q = 0; q < QM; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int p = 0; p < QN; ++p) {
                    const float *v = &acc[q * 4 + i][p * 4];
                    *reinterpret_cast<float4 *>(smem + (q * SUBM + tm2 * 4 + i) * PITCH +
                                                p * SUBN + tn2 * 4) =
                        make_float4(v[0], v[1], v[2], v[3]);
                }
        cluster_sync();
        switch (gridDim.y) {  // S: 1 (a cluster of one), 2, 4 or 8
        case 2: cluster_add_partials<BM, BN, PITCH, C_VEC, 2>(smem, M, N, C, (int)aux); break;
        case 4: cluster_add_partials<BM, BN, PITCH, C_VEC, 4>(smem, M, N, C, (int)aux); break;
        case 8: cluster_add_partials<BM, BN, PITCH, C_VEC, 8>(smem, M, N, C, (int)aux); break;
        default: cluster_add_partials<BM, BN, PITCH, C_VEC, 1>(smem, M, N, C, (int)aux); break;
        }
        cluster_sync();
    } else {
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
}

// Shared memory a cluster-split CTA reserves to have an SM to itself: more
// than half of the 228 KB an SM holds.
constexpr size_t kSpreadSmemBytes = 120 * 1024;

template <int BM, int BN, int BK, int STAGES, int MINB, int ORDER, bool B_VEC, bool C_VEC,
          int SPLIT>
// tile_first / tile_count: launch only tiles tile_first .. +tile_count - 1 of
// the grouped raster (tile_count < 0: all from tile_first on); a plain or
// workspace grid must start at tile 0.
cudaError_t launch_cfg(int M, int N, int K, const float *A, const float *B, float *C,
                       cudaStream_t stream, int splits = 1, int kchunk = 0, bool spread = false,
                       long long tile_first = 0, long long tile_count = -1)
{
    static_assert(Cfg<BM, BN, BK, STAGES>::CLUSTER_SMEM_BYTES <= kSpreadSmemBytes,
                  "the spread reservation holds the pipeline and the partial tile");
    using G = Cfg<BM, BN, BK, STAGES>;
    auto kernel = sgemm_rt_kernel<BM, BN, BK, STAGES, MINB, ORDER, B_VEC, C_VEC, SPLIT>;
    // A cluster split may ask for one CTA per SM (spread): it then reserves
    // more shared memory than two CTAs of an SM could hold.
    constexpr size_t smem_max = SPLIT == kSplitCluster ? kSpreadSmemBytes : G::SMEM_BYTES;
    const size_t smem = SPLIT != kSplitCluster ? G::SMEM_BYTES
                        : spread               ? kSpreadSmemBytes
                                               : G::CLUSTER_SMEM_BYTES;
    if (smem_max > 48 * 1024) {
        static std::atomic<uint64_t> done{0};  // per instantiation
        const cudaError_t e = set_smem_limit_once(kernel, (int)smem_max, done);
        if (e != cudaSuccess)
            return e;
    }
    const long long all_tiles = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    if (all_tiles > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    if (tile_first < 0 || tile_first > all_tiles || (SPLIT != kSplitCluster && tile_first != 0))
        return cudaErrorInvalidValue;
    const long long tiles = tile_count < 0 || tile_first + tile_count > all_tiles
                                ? all_tiles - tile_first
                                : tile_count;
    if (tiles == 0)
        return cudaSuccess;
    if (splits < 1 || splits > 65535 || (SPLIT == kPlain && splits != 1))
        return cudaErrorInvalidValue;
    if (splits == 1)
        kchunk = K;
    if constexpr (SPLIT == kSplitCluster) {
        // S = splits CTAs per cluster, S dividing BM (S in 1, 2, 4, 8).
        if (splits > 8 || BM % splits != 0)
            return cudaErrorInvalidValue;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)tiles, (unsigned)splits, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = (unsigned)splits;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, M, N, K, kchunk, A, B, C, (size_t)tile_first);
    }
    kernel<<<dim3((unsigned)tiles, (unsigned)splits), kThreads, smem, stream>>>(
        M, N, K, kchunk, A, B, C, (size_t)M * N);
    return cudaGetLastError();
}

template <int BM, int BN, int BK, int STAGES, int MINB, int ORDER, int SPLIT = kPlain>
cudaError_t launch_any(int M, int N, int K, const float *A, const float *B, float *C,
                       cudaStream_t stream, int splits = 1, int kchunk = 0, bool spread = false,
                       long long tile_first = 0, long long tile_count = -1)
{
    const bool b_vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(B) & 15) == 0);
    const bool c_vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15) == 0);
    // Three instantiations: the 4-byte B path (rows not 16-byte aligned) also
    // takes the 4-byte C stores.
    if (b_vec && c_vec)
        return launch_cfg<BM, BN, BK, STAGES, MINB, ORDER, true, true, SPLIT>(
            M, N, K, A, B, C, stream, splits, kchunk, spread, tile_first, tile_count);
    if (b_vec)
        return launch_cfg<BM, BN, BK, STAGES, MINB, ORDER, true, false, SPLIT>(
            M, N, K, A, B, C, stream, splits, kchunk, spread, tile_first, tile_count);
    return launch_cfg<BM, BN, BK, STAGES, MINB, ORDER, false, false, SPLIT>(
        M, N, K, A, B, C, stream, splits, kchunk, spread, tile_first, tile_count);
}

} // namespace simt

namespace {
using namespace simt_tiles;

__global__ void splitk_reduce_kernel(const float *__restrict__ W, float *__restrict__ C,
                                     int64_t count, int splits)
{
    // C[i] = W[0][i] + W[1][i] + ... in increasing split order (deterministic).
    grid_dependency_wait();  // launched as a programmatic dependent of the split kernel
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
        float s = W[i];
        for (int t = 1; t < splits; ++t)
            s += W[(int64_t)t * count + i];
        C[i] = s;
    }
}

__global__ void splitk_reduce4_kernel(const float4 *__restrict__ W, float4 *__restrict__ C,
                                      int64_t count4, int splits)
{
    grid_dependency_wait();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count4; i += stride) {
        float4 s = W[i];
        for (int t = 1; t < splits; ++t) {
            const float4 v = W[(int64_t)t * count4 + i];
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        C[i] = s;
    }
}
} // namespace

namespace {

// 256 x 64 tiles for tall, narrow products. Only the 16-byte B path is built
// for them (its 4-byte variant spilled registers under the 128-register
// budget); rows of B off 16-byte boundaries take 128 x 64 tiles with the same
// split, packed two CTAs to an SM.
template <int SPLIT>
cudaError_t launch_tall(int M, int N, int K, const float *A, const float *B, float *C,
                        cudaStream_t stream, int splits = 1, int kchunk = 0, bool spread = false)
{
    const bool b_vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(B) & 15) == 0);
    const bool c_vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15) == 0);
    if (!b_vec)
        return simt::launch_any<kTileM, kNarrowN, kSliceK, 2, 2, 1, SPLIT>(M, N, K, A, B, C, stream,
                                                                         splits, kchunk, false);
    if (c_vec)
        return simt::launch_cfg<kTallTileM, kNarrowN, kSliceK, 2, 2, 1, true, true, SPLIT>(
            M, N, K, A, B, C, stream, splits, kchunk, spread);
    return simt::launch_cfg<kTallTileM, kNarrowN, kSliceK, 2, 2, 1, true, false, SPLIT>(
        M, N, K, A, B, C, stream, splits, kchunk, spread);
}

// The SIMT kernel on tile shape `tile` (resolved: both sides set), plain or
// with K split over the CTAs of a cluster.
template <int SPLIT>
cudaError_t launch_tile(SimtTile tile, int M, int N, int K, const float *A, const float *B,
                        float *C, cudaStream_t stream, int splits = 1, int kchunk = 0,
                        bool spread = false)
{
    if (tile.m == kTallTileM && tile.n == kNarrowN)
        return launch_tall<SPLIT>(M, N, K, A, B, C, stream, splits, kchunk, spread);
    if (tile.m == kShortTileM && tile.n == kWideTileN)  // 4 x 16 per thread
        return simt::launch_any<kShortTileM, kWideTileN, kSliceK, 2, 2, 1, SPLIT>(
            M, N, K, A, B, C, stream, splits, kchunk, spread);
    if (tile.m == kShortTileM && tile.n == kNarrowN)
        return simt::launch_any<kShortTileM, kNarrowN, kSliceK, 2, 2, 1, SPLIT>(
            M, N, K, A, B, C, stream, splits, kchunk, spread);
    if (tile.m == kShortTileM)
        return simt::launch_any<kShortTileM, kTileN, kSliceK, 2, 2, 1, SPLIT>(
            M, N, K, A, B, C, stream, splits, kchunk, spread);
    if (tile.n == kNarrowN)
        return simt::launch_any<kTileM, kNarrowN, kSliceK, 2, 2, 1, SPLIT>(
            M, N, K, A, B, C, stream, splits, kchunk, spread);
    return simt::launch_any<kTileM, kTileN, kSliceK, 2, 2, 1, SPLIT>(M, N, K, A, B, C, stream,
                                                                   splits, kchunk, spread);
}

} // namespace

cudaError_t launch_sgemm_f32(int M, int N, int K, const float *A, const float *B, float *C,
                             cudaStream_t stream, SimtTile tile, const SimtTma *tma)
{
    // Without a choice, 64-row tiles for M <= 64 (128-row tiles would be at
    // least half empty) and 64-column tiles for N <= 64.
    const SimtTile t = simt_resolve_tile(tile, M, N);
    if (tma && t.m == kTileM && t.n == kTileN && sgemm_tma_eligible(M, N, K, A, B, tma->lda, tma->ldb))
        return launch_sgemm_f32_tma(M, N, K, A, B, C, *tma, -1, stream);
    if (tma && ((t.m == kTallTileM && t.n == kNarrowN) || (t.m == kShortTileM && t.n == kWideTileN)) &&
        sgemm_tma_eligible(M, N, K, A, B, tma->lda, tma->ldb))
        return launch_sgemm_f32_tma_rect(t, M, N, K, A, B, C, *tma, 1,
                                         (K + kSliceK - 1) / kSliceK * kSliceK, false, stream);
    return launch_tile<simt::kPlain>(t, M, N, K, A, B, C, stream);
}

cudaError_t launch_sgemm_f32_splitk(int M, int N, int K, const float *A, const float *B, float *C,
                                    const SplitK &plan, float *workspace, cudaStream_t stream)
{
    using simt::kSplitWorkspace;
    cudaError_t e;
    if (M <= kShortTileM)
        e = N <= kNarrowN
                ? simt::launch_any<kShortTileM, kNarrowN, kSliceK, 2, 2, 1, kSplitWorkspace>(
                      M, N, K, A, B, workspace, stream, plan.splits, plan.kchunk)
                : simt::launch_any<kShortTileM, kTileN, kSliceK, 2, 2, 1, kSplitWorkspace>(
                      M, N, K, A, B, workspace, stream, plan.splits, plan.kchunk);
    else
        e = N <= kNarrowN
                ? simt::launch_any<kTileM, kNarrowN, kSliceK, 2, 2, 1, kSplitWorkspace>(
                      M, N, K, A, B, workspace, stream, plan.splits, plan.kchunk)
                : simt::launch_any<kTileM, kTileN, kSliceK, 2, 2, 1, kSplitWorkspace>(
                      M, N, K, A, B, workspace, stream, plan.splits, plan.kchunk);
    if (e != cudaSuccess)
        return e;
    const int64_t count = (int64_t)M * N;
    const bool vec = (count % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(workspace) & 15) == 0);
    const int64_t items = vec ? count / 4 : count;
    int64_t blocks = (items + 255) / 256;
    if (blocks > 4096)
        blocks = 4096;
    // A programmatic dependent of the split kernel: launched while the partial
    // products are still being computed, it waits for them in the kernel.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (vec)
        return cudaLaunchKernelEx(&cfg, splitk_reduce4_kernel,
                                  reinterpret_cast<const float4 *>(workspace),
                                  reinterpret_cast<float4 *>(C), count / 4, plan.splits);
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, (const float *)workspace, C, count,
                              plan.splits);
}

int sgemm_cluster_resident_spread(int cluster_size)
{
    // Every cluster-split instantiation has the same footprint when spread
    // (256 threads, at most 128 registers, kSpreadSmemBytes), so one of them
    // stands for all in the occupancy query.
    auto kernel = simt::sgemm_rt_kernel<kTileM, kTileN, kSliceK, 2, 2, 1, true, true,
                                        simt::kSplitCluster>;
    static std::atomic<uint64_t> done{0};
    if (set_smem_limit_once(kernel, (int)simt::kSpreadSmemBytes, done) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (cluster_size != 2 && cluster_size != 4 && cluster_size != 8)
        return 0;
    static std::atomic<int> cache2[64] = {}, cache4[64] = {}, cache8[64] = {};
    auto &cache = cluster_size == 2 ? cache2 : cluster_size == 4 ? cache4 : cache8;
    return resident_clusters(kernel, cluster_size, simt::kThreads, simt::kSpreadSmemBytes, cache);
}

SplitK sgemm_cluster_schedule(int M, int N, int K, int sm_count, double *est)
{
    // The fewest tiles any candidate tile shape gives (256 x 64 for tall,
    // narrow products, 64 x 256 for short ones).
    const int tile_n = N <= kNarrowN ? kNarrowN : M <= kShortTileM ? kWideTileN : kTileN;
    const int tile_m = M <= kShortTileM ? kShortTileM : N <= kNarrowN ? kTallTileM : kTileM;
    const long long tiles = (long long)((M + tile_m - 1) / tile_m) * ((N + tile_n - 1) / tile_n);
    int resident[3] = {0, 0, 0};
    if (tiles <= sm_count)  // only then is a split considered
        for (int i = 0; i < 3; ++i)
            resident[i] = sgemm_cluster_resident_spread(2 << i);
    return sgemm_cluster_plan(M, N, K, sm_count, resident, est);
}

F32Schedule sgemm_ws_schedule(int M, int N, int K, int sm_count)
{
    double cluster_est = 0, streamk_est = 1e300;
    F32Schedule f;
    f.workspace = sgemm_splitk_plan(M, N, K, sm_count);
    f.cluster = sgemm_cluster_schedule(M, N, K, sm_count, &cluster_est);
    const double ws_est = sgemm_workspace_estimate(M, N, K, sm_count, f.workspace);
    if (f.workspace.splits > 1 && cluster_est < ws_est)
        f.workspace = SplitK{1, K};
    const int sk = sgemm_streamk_plan(M, N, K, sm_count, &streamk_est);
    if (sk > 0 && streamk_est < cluster_est && (f.workspace.splits <= 1 || streamk_est < ws_est)) {
        f.streamk = sk;
        f.workspace = SplitK{1, K};
    }
    return f;
}

cudaError_t launch_sgemm_f32_cluster(int M, int N, int K, const float *A, const float *B, float *C,
                                     const SplitK &plan, cudaStream_t stream, const SimtTma *tma)
{
    const SimtTile t = simt_resolve_tile(plan.tile, M, N);
    if (tma && t.m == kTileM && t.n == kTileN && sgemm_tma_eligible(M, N, K, A, B, tma->lda, tma->ldb))
        return launch_sgemm_f32_tma_cluster(M, N, K, A, B, C, *tma, plan.splits, plan.kchunk,
                                            plan.spread, 0, -1, stream);
    if (tma && ((t.m == kTallTileM && t.n == kNarrowN) || (t.m == kShortTileM && t.n == kWideTileN)) &&
        sgemm_tma_eligible(M, N, K, A, B, tma->lda, tma->ldb))
        return launch_sgemm_f32_tma_rect(t, M, N, K, A, B, C, *tma, plan.splits, plan.kchunk,
                                         plan.spread, stream);
    return launch_tile<simt::kSplitCluster>(t, M, N, K, A, B, C, stream, plan.splits, plan.kchunk,
                                            plan.spread);
}

cudaError_t launch_sgemm_f32_tail(int M, int N, int K, const float *A, const float *B, float *C,
                                  const TailPlan &plan, cudaStream_t stream, const SimtTma *tma)
{
    using simt::kSplitCluster;
    if (M <= kShortTileM || N <= kNarrowN || plan.tail.splits < 2)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaSuccess;
    const bool use_tma = tma && sgemm_tma_eligible(M, N, K, A, B, tma->lda, tma->ldb);
    if (plan.plain_tiles > 0 && use_tma)
        e = launch_sgemm_f32_tma(M, N, K, A, B, C, *tma, plan.plain_tiles, stream);
    else if (plan.plain_tiles > 0)
        e = simt::launch_any<kTileM, kTileN, kSliceK, 2, 2, 1>(M, N, K, A, B, C, stream, 1, 0, false,
                                                               0, plan.plain_tiles);
    if (e != cudaSuccess)
        return e;
    if (use_tma)
        return launch_sgemm_f32_tma_cluster(M, N, K, A, B, C, *tma, plan.tail.splits,
                                            plan.tail.kchunk, false, plan.plain_tiles, -1, stream);
    return simt::launch_any<kTileM, kTileN, kSliceK, 2, 2, 1, kSplitCluster>(
        M, N, K, A, B, C, stream, plan.tail.splits, plan.tail.kchunk, false, plan.plain_tiles);
}

bool sgemm_tiles_use_tma(int M, int N, int K, const SplitK &cluster, int sm_count)
{
    const SimtTile t = simt_resolve_tile(cluster.tile, M, N);
    const bool tma_tile = (t.m == kTileM && t.n == kTileN) || (t.m == kTallTileM && t.n == kNarrowN) ||
                          (t.m == kShortTileM && t.n == kWideTileN);
    if (cluster.splits > 1)
        return tma_tile;
    if (sgemm_tail_plan(M, N, K, sm_count).tail.splits > 1)
        return true;  // 128 x 128 tiles
    return tma_tile;
}

cudaError_t launch_sgemm_f32_tiles(int M, int N, int K, const float *A, const float *B, float *C,
                                   const SplitK &cluster, int sm_count, cudaStream_t stream,
                                   const SimtTma *tma)
{
    if (cluster.splits > 1)
        return launch_sgemm_f32_cluster(M, N, K, A, B, C, cluster, stream, tma);
    const TailPlan tail = sgemm_tail_plan(M, N, K, sm_count);
    if (tail.tail.splits > 1)
        return launch_sgemm_f32_tail(M, N, K, A, B, C, tail, stream, tma);
    return launch_sgemm_f32(M, N, K, A, B, C, stream, cluster.tile, tma);
}

} // namespace rtm
