// Internal launch functions shared between the C-ABI translation unit and the
// kernel translation units. Arguments are already validated by the caller.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

namespace rtm {

// Raise `kernel`'s dynamic shared-memory limit to `bytes` the first time it is
// launched on the current device. `done` is one bit per device (a static of
// the call site); concurrent first callers may both set the attribute, which
// is harmless, and no flag is read or written without atomics.
// With `carveout_pct` >= 0 it also states the preferred shared-memory
// carve-out (percent of the SM's maximum), so that kernels whose loads pass
// through L1 leave it the rest of the SM's unified memory.
template <typename Kernel>
cudaError_t set_smem_limit_once(Kernel kernel, int bytes, std::atomic<uint64_t> &done,
                                int carveout_pct = -1)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit))
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && carveout_pct >= 0)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 carveout_pct);
    if (e == cudaSuccess && bit)
        done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Tiles of the SIMT FP32 product: 128 x 128 C tiles, with 64 columns for
// N <= 64 and 64 rows for M <= 64 (where 128 would be at least half empty),
// 32-deep K slices. Tall, narrow products (N <= 64, M > 128) may take 256 x 64
// tiles instead (16 x 4 outputs per thread: fewer shared reads per FMA than
// the 8 x 4 of a 128 x 64 tile), and products with 64 rows or fewer 64 x 256
// tiles (4 x 16 per thread against the 4 x 8 of a 64 x 128 tile), where the
// schedule model prices them lower.
namespace simt_tiles {
constexpr int kTileM = 128, kTileN = 128, kSliceK = 32;
constexpr int kNarrowN = 64;
constexpr int kShortTileM = 64;
constexpr int kTallTileM = 256;
constexpr int kWideTileN = 256;
} // namespace simt_tiles

// Tile shape of a SIMT schedule, rows x columns of C per CTA: 128 x 128,
// 128 x 64, 64 x 128, 64 x 64, 256 x 64 or 64 x 256. {0, 0} stands for the
// standard shape of the product (simt_standard_tile).
struct SimtTile {
    int m = 0, n = 0;
};
inline SimtTile simt_standard_tile(int M, int N)
{
    return SimtTile{M <= simt_tiles::kShortTileM ? simt_tiles::kShortTileM : simt_tiles::kTileM,
                    N <= simt_tiles::kNarrowN ? simt_tiles::kNarrowN : simt_tiles::kTileN};
}
inline SimtTile simt_resolve_tile(SimtTile t, int M, int N)
{
    return t.m > 0 && t.n > 0 ? t : simt_standard_tile(M, N);
}

// How many clusters of `cluster_size` CTAs of `kernel` (`threads` threads,
// `smem` bytes of dynamic shared memory, attribute already set) can be
// resident at once on the current device; cached in `cache` (one slot per
// device). 0 if the query fails. Kernels whose CTAs wait for each other at a
// cluster barrier use it to launch no more clusters than fit at once: a
// cluster that must wait for another to finish doubles the time.
template <typename Kernel>
int resident_clusters(Kernel kernel, int cluster_size, int threads, size_t smem,
                      std::atomic<int> (&cache)[64])
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 0;
    }
    int n = cache[dev].load();
    if (n > 0)
        return n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cluster_size, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster_size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 0;
    }
    cache[dev].store(n);
    return n;
}

// What the TMA-fed SIMT kernel needs from the caller: the driver's
// cuTensorMapEncodeTiled, the device error word its bounded waits report to,
// and the wait limit.
struct SimtTma {
    void *encode_tiled = nullptr;
    int *err = nullptr;
    uint64_t wait_limit_ns = 0;
    bool mute = false;  // failure-detection self-test: announce the slices, load nothing
    // Row strides of A and B in elements (0: K and N), for operands re-pitched
    // into a workspace; read only by the tensor maps.
    int64_t lda = 0, ldb = 0;
};
// The plain 128 x 128 product with its K slices loaded by TMA (sgemm_tma.cu):
// tiles 0 .. tile_count - 1 of the grouped raster (tile_count < 0: all).
// Needs sgemm_tma_eligible: row strides of A and B (lda, ldb; 0: K and N)
// multiples of 4 elements, A and B 16-byte aligned. Same sums in the same
// order as the cp.async kernel (same bits).
bool sgemm_tma_eligible(int M, int N, int K, const float *A, const float *B, int64_t lda = 0,
                        int64_t ldb = 0);
// mute: the failure-detection self-test (no loads are issued; every bounded
// wait runs out; C is left unspecified).
cudaError_t launch_sgemm_f32_tma(int M, int N, int K, const float *A, const float *B, float *C,
                                 const SimtTma &tma, long long tile_count, cudaStream_t stream,
                                 bool mute = false);

// The same tiles with K split over `splits` (1, 2, 4 or 8) CTAs of a cluster,
// kchunk of K each (a multiple of 32), the partial tiles added through
// distributed shared memory in rank order; tiles tile_first .. +tile_count - 1
// (tile_count < 0: to the end); spread: one CTA per SM (sgemm_tma.cu).
cudaError_t launch_sgemm_f32_tma_cluster(int M, int N, int K, const float *A, const float *B,
                                         float *C, const SimtTma &tma, int splits, int kchunk,
                                         bool spread, long long tile_first, long long tile_count,
                                         cudaStream_t stream);
// The same TMA-fed loop on rectangular tiles (sgemm_tma_rect.cu): `tile` 256 x 64
// (16 x 4 outputs per thread, tall, narrow products) or 64 x 256 (4 x 16,
// products of 33-64 rows), K split over `splits` (1, 2, 4 or 8) CTAs of a
// cluster in chunks of `kchunk` (a multiple of 32, splits * kchunk >= K);
// spread: one CTA per SM. Same operand rules as launch_sgemm_f32_tma.
cudaError_t launch_sgemm_f32_tma_rect(SimtTile tile, int M, int N, int K, const float *A,
                                      const float *B, float *C, const SimtTma &tma, int splits,
                                      int kchunk, bool spread, cudaStream_t stream);
// Stream-K over the TMA-fed 128 x 128 tiles (sgemm_tma.cu): `ctas` CTAs take
// equal ranges of the tiles x K-slices iterations; tiles split between CTAs
// are added by a fixup kernel in a fixed order (repeatable bit for bit).
// workspace: sgemm_streamk_workspace_floats(M, N, ctas) floats, 16-byte
// aligned. Operands as launch_sgemm_f32_tma. spread: one CTA per SM.
int64_t sgemm_streamk_workspace_floats(int M, int N, int ctas);
cudaError_t launch_sgemm_f32_streamk(int M, int N, int K, const float *A, const float *B, float *C,
                                     const SimtTma &tma, int ctas, bool spread, float *workspace,
                                     cudaStream_t stream);

// SIMT FP32 register-tiled product (sgemm_simt.cu): any shape and
// 4-byte-aligned pointers. 1 <= K; M, N >= 1. `tile`: the CTA tile shape
// (any of SimtTile's; 256 x 64 tiles are taken only when the rows of B lie on
// 16-byte boundaries, 128 x 64 otherwise). With `tma` set, 128 x 128 tiles of
// operands sgemm_tma_eligible accepts run on the TMA-fed kernel.
cudaError_t launch_sgemm_f32(int M, int N, int K, const float *A, const float *B, float *C,
                             cudaStream_t stream, SimtTile tile = SimtTile{},
                             const SimtTma *tma = nullptr);

// SIMT FP32 product for short, wide shapes (sgemm_short.cu): M <= kShortMaxM,
// any N and K >= 1, 4-byte-aligned pointers. Each thread keeps one column of
// C in registers; `splits` (1, 2, 4 or 8, from sgemm_short_splits) CTAs of a
// cluster split K and add their partials in rank order. No workspace.
constexpr int kShortMaxM = 32;
int sgemm_short_splits(int M, int N, int K, int sm_count);
cudaError_t launch_sgemm_short(int M, int N, int K, const float *A, const float *B, float *C,
                               int splits, cudaStream_t stream);

// Split-K schedule of the SIMT product for shapes with too few C tiles to
// fill the GPU: `splits` CTA rows each sum `kchunk` of K (a multiple of the
// 32-deep slice) into their own M x N slab of a workspace, then a reduction
// kernel adds the slabs in increasing split order (deterministic).
struct SplitK {
    int splits;  // 1: no split (plain product)
    int kchunk;
    bool spread = false;  // cluster split: one CTA per SM (see sgemm_cluster_plan)
    SimtTile tile{};  // set by sgemm_cluster_plan only ({0, 0}: the standard shape)
};
SplitK sgemm_splitk_plan(int M, int N, int K, int sm_count);  // sgemm_plan.cu
// The plan's run time in the slice-time units of sgemm_cluster_plan's
// estimate, for choosing between the two splits (1e300 when not split).
double sgemm_workspace_estimate(int M, int N, int K, int sm_count, const SplitK &plan);
// workspace: plan.splits * M * N floats. 1 <= K; M, N >= 1; plan.splits >= 2.
cudaError_t launch_sgemm_f32_splitk(int M, int N, int K, const float *A, const float *B, float *C,
                                    const SplitK &plan, float *workspace, cudaStream_t stream);
// Split-K without a workspace: the plan.splits (2, 4 or 8) CTAs that share a C
// tile form one cluster and add their partial tiles through distributed shared
// memory in rank order (deterministic). plan.splits == 1 is the plain product.
// plan.tile: the tile shape the product (split or not) runs on. *est: the
// chosen schedule's estimate (also for an unsplit product).
// resident_spread[i]: clusters of 2 << i CTAs that fit at once with one CTA
// per SM (sgemm_cluster_resident_spread; 0 if unknown).
SplitK sgemm_cluster_plan(int M, int N, int K, int sm_count, const int (&resident_spread)[3],
                          double *est = nullptr);  // sgemm_plan.cu
int sgemm_cluster_resident_spread(int cluster_size);
// sgemm_cluster_plan with the current device's cluster residency.
SplitK sgemm_cluster_schedule(int M, int N, int K, int sm_count, double *est = nullptr);
// Products with more tiles than SMs: tiles 0 .. plain_tiles - 1 run as the
// plain product, the rest with K split over clusters (tail.splits > 1; none
// when tail.splits == 1). sgemm_plan.cu.
struct TailPlan {
    long long plain_tiles;
    SplitK tail;
};
TailPlan sgemm_tail_plan(int M, int N, int K, int sm_count);
cudaError_t launch_sgemm_f32_tail(int M, int N, int K, const float *A, const float *B, float *C,
                                  const TailPlan &plan, cudaStream_t stream,
                                  const SimtTma *tma = nullptr);
// Whether launch_sgemm_f32_tiles runs this schedule on TMA-fed kernels when
// the operands allow it (128 x 128, 256 x 64 or 64 x 256 tiles, or the tail
// split); otherwise it runs the cp.async kernels, which read A and B with row
// strides K and N.
bool sgemm_tiles_use_tma(int M, int N, int K, const SplitK &cluster, int sm_count);
// The register-tiled product on its own schedule: K split over clusters when
// cluster.splits > 1, else the tail plan, else the plain product (its
// unsplit 128 x 128 tiles on the TMA-fed kernel when `tma` is set and the
// operands allow it).
cudaError_t launch_sgemm_f32_tiles(int M, int N, int K, const float *A, const float *B, float *C,
                                   const SplitK &cluster, int sm_count, cudaStream_t stream,
                                   const SimtTma *tma = nullptr);
// How gemm_f32_ws (and gemm_f32_noalloc) schedule a product with M > kShortMaxM:
// the workspace split when the model prices it below the cluster split (ties
// go to the workspace), else the cluster split or the plain product.
struct F32Schedule {
    SplitK workspace;  // splits > 1: split-K through a workspace of splits * M * N floats
    SplitK cluster;    // used when workspace.splits == 1 and streamk == 0
    int streamk = 0;   // > 0: stream-K over this many CTAs (launch_sgemm_f32_streamk)
};
// Stream-K's CTA count for a product (0: not a stream-K product: 64-row or
// 64-column tiles, or more 128 x 128 tiles than SMs) and, in *est, its run
// time in the slice-time units of sgemm_cluster_plan's estimate. sgemm_plan.cu.
int sgemm_streamk_plan(int M, int N, int K, int sm_count, double *est);
F32Schedule sgemm_ws_schedule(int M, int N, int K, int sm_count);
cudaError_t launch_sgemm_f32_cluster(int M, int N, int K, const float *A, const float *B, float *C,
                                     const SplitK &plan, cudaStream_t stream,
                                     const SimtTma *tma = nullptr);

// The page's ablation ladder (sgemm_ladder.cu): rung 0 naive, 1 shared-memory
// tiled (TILE 32), 2 register tiled (64 x 64 block, 4 x 4 per thread).
cudaError_t launch_sgemm_ladder(int rung, int M, int N, int K, const float *A, const float *B,
                                float *C, cudaStream_t stream);

// tcgen05 bf16 x bf16 (or fp16 x fp16) -> fp32 product (gemm_tc.cu). K >= 1, K % 8 == 0,
// N % 8 == 0, A/B/C 16-byte aligned. `err` is the device error word;
// `wait_limit_ns` bounds every wait; `mute_producer` != 0 issues no loads
// (failure-detection self-test only).
struct TcLaunch {
    int M, N, K;
    const uint16_t *A;
    const uint16_t *B;
    float *C;
    int *err;
    uint64_t wait_limit_ns;
    int mute_producer;
    int sm_count;
    void *encode_tiled;  // cuTensorMapEncodeTiled driver entry point
    int f16;             // 0: A and B are bf16; 1: A and B are fp16
    int64_t lda = 0;     // row stride of A in elements (0: K); CTA-pair kernel only
    int64_t ldb = 0;     // row stride of B in elements (0: N); CTA-pair kernel only
};
// The single-CTA kernel with 128 x bn tiles, bn in {256, 128, 64} (narrower
// tiles give short, wide products more CTAs).
cudaError_t launch_gemm_bf16_tc_bn(const TcLaunch &p, int bn, cudaStream_t stream);
// The same product on CTA pairs (gemm_tc2.cu, tcgen05 cta_group::2, 256 x 256
// tiles); used for M > 128, where a pair tile is not mostly empty. A and B
// rows at lda / ldb elements (16-byte multiples, 16-byte aligned bases); any
// 4-byte-aligned C and any N (float4 stores when C rows are 16-byte aligned).
cudaError_t launch_gemm_tc_pair(const TcLaunch &p, cudaStream_t stream);
// splits 1 or 2 (2: C zero-filled, then each K half reduce-added; C rows must be
// 16-byte aligned); 0 lets the launcher choose (launch_gemm_tc_pair).
cudaError_t launch_gemm_tc_pair_split(const TcLaunch &p, int splits, cudaStream_t stream);
// The first of `ntiles` pair tiles whose K is split in two when `pairs` CTA
// pairs are resident and K has `kblocks` 64-deep blocks (ntiles: none). tc_plan.cu.
long long pair_split_from(long long ntiles, int pairs, int kblocks, bool c_vec);

// Copy a rows x cols matrix of 2-byte values (row-major, rows packed, `src`
// 2-byte aligned) to `dst` with rows `ld` values apart (ld >= cols, ld % 8 ==
// 0, dst 16-byte aligned), so that every row starts on a 16-byte boundary
// (pack.cu). Values in columns cols .. ld-1 of dst are unspecified.
cudaError_t launch_pack_rows_2b(const uint16_t *src, int64_t rows, int64_t cols, uint16_t *dst,
                                int64_t ld, int sm_count, cudaStream_t stream);
// The same for 4-byte values (fp32): ld a multiple of 4 elements.
cudaError_t launch_pack_rows_4b(const float *src, int64_t rows, int64_t cols, float *dst,
                                int64_t ld, int sm_count, cudaStream_t stream);
// Products with one short side and K split over CTA clusters (gemm_tc_t.cu).
// swap: short, wide products as C^T = B^T.A^T, CTAs own 128 columns of C and
// tct_rows(M) (32, 64 or 128) rows. No swap: tall, narrow products, CTAs own
// 128 rows and tcs_cols(N) (64 or 128) columns. `splits` (1, 2, 4 or 8)
// CTAs of a cluster split K and sum their partial tiles in rank order. Same
// operand rules as launch_gemm_bf16_tc_bn (rows on 16-byte boundaries).
int tct_rows(int M);
int tcs_cols(int N);
cudaError_t launch_gemm_tc_t(const TcLaunch &p, int splits, bool swap, cudaStream_t stream);
// The K-split of those kernels for `tiles` 128-wide tiles (tc_plan.cu): 0 when
// K has fewer than 32 64-deep blocks or the tiles outnumber the SMs, else the
// largest S in {1, 2, 4, 8} with tiles * S <= sms and >= 16 blocks per CTA.
int long_k_splits(long long tiles, long long K, int sms);
// The CTA-pair product for any K, N and 2-byte-aligned A, B (gemm_tc_any.cu;
// 256 x 256 tiles, each CTA staging half of the operands), for M > 128:
// operands loaded by producer warps instead of TMA (mute_producer: they load
// nothing, so every wait gives up); any 4-byte-aligned C.
cudaError_t launch_gemm_tc_any_pair(const TcLaunch &p, cudaStream_t stream);
// launch_gemm_tc_t's two tilings with producer warps instead of TMA
// (gemm_tc_any_t.cu): with swap, short products (M <= 128), CTAs own 128
// columns and tct_rows(M) rows; without, tall, narrow products (N <= 128),
// CTAs own 128 rows and tcs_cols(N) columns. `splits` (1, 2, 4 or 8) CTAs of a
// cluster split K; with splits = 1 the tiles may outnumber the SMs (several
// waves). Same operand rules as launch_gemm_tc_any_pair.
cudaError_t launch_gemm_tc_any_t(const TcLaunch &p, int splits, bool swap, cudaStream_t stream);

// The host-side argument checks of the fp32 entry points (api.cu), made
// before any CUDA call: GEMM_OK with *nothing_to_do set when M or N is zero,
// else GEMM_OK or the status the entry points return for these arguments.
int check_f32_args(int64_t M, int64_t N, int64_t K, const float *A, const float *B, const float *C,
                   bool *nothing_to_do);

// C[0 .. count) = 0 (the K == 0 product).
cudaError_t launch_zero_fill(float *C, int64_t count, cudaStream_t stream);

// Status codes written into the device error word (same values as gemm.h).
constexpr int kDevErrTimeout = -4;

} // namespace rtm
