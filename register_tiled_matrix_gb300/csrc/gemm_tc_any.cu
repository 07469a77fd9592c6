// bf16/fp16 -> fp32 product C = A.B on tcgen05 for any shape and any 2-byte
// aligned pointers: the path for rows that do not start on 16-byte
// boundaries (K % 8 != 0 or N % 8 != 0, or offset pointers), which the
// tensor-memory-access unit cannot address.
//
// Same tiling and accumulator handling as the single-CTA kernel of
// gemm_tc.cu (128 x 256 tiles, 64-deep K-slices, a 4-stage ring, tcgen05.mma
// kind::f16 M 128 N 256 K 16 into double-buffered tensor memory, bounded
// waits), with the TMA producer replaced by eight producer warps that load
// the A and B slices with plain 2-byte loads and store them into the same
// 128-byte-swizzled shared-memory layouts the MMA descriptors describe
// (16-byte chunk c of a 128-byte row r at chunk c ^ (r mod 8)), writing zeros
// outside M, N, K. Each producer thread then makes its shared-memory writes
// visible to the tensor core (fence.proxy.async) and arrives on the stage's
// barrier. The epilogue stores scalars where C rows are not 16-byte aligned.
//
// Loads and stores move V consecutive values at once (V = 1, 2 or 4: 2-, 4-
// or 8-byte accesses), the largest V for which every row of A and B starts on
// a 2V-byte boundary (K and N multiples of V, A and B 2V-byte aligned), so a
// vector never straddles a row end or a 16-byte swizzle chunk. With 8-byte
// access the producers issue cp.async copies straight into the swizzled
// layout and keep three K-slices in flight; the narrower paths stage the
// values in registers, one K-slice at a time.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace rtm {
namespace tcany {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int UMMA_K = 16;
constexpr int kProducerWarps = 8;
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kMmaWarp = kProducerWarps;               // warp 8
constexpr int kFirstEpilogueWarp = kProducerWarps + 1;  // warps 9..12 (quarters 1,2,3,0)
constexpr int kThreads = (kProducerWarps + 1 + 4) * 32;
constexpr int kGroupM = 16;
constexpr int kAsyncDepth = 3;  // K-slices in flight per producer thread (cp.async path)
constexpr uint32_t A_STAGE_BYTES = BM * BK * 2;
constexpr uint32_t B_ATOM_BYTES = BK * 64 * 2;
constexpr uint32_t B_STAGE_BYTES = BK * BN * 2;
constexpr uint32_t STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr size_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;

template <bool F16>
__host__ __device__ constexpr uint32_t idesc()
{
    return (1u << 4) | ((F16 ? 0u : 1u) << 7) | ((F16 ? 0u : 1u) << 10) | (0u << 15) |
           (1u << 16) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

struct Params {
    int M, N, K;
    const uint16_t *A;
    const uint16_t *B;
    float *C;
    int *err;
    unsigned long long limit_ns;
};

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

// Byte offset of element (row, col) in a 128-byte-swizzled tile of 64-element
// rows (one row = 128 bytes; the tile base is 1024-byte aligned).
__device__ __forceinline__ uint32_t swz(int row, int col)
{
    return (uint32_t)row * 128u + ((((uint32_t)col >> 3) ^ ((uint32_t)row & 7u)) << 4) +
           ((uint32_t)col & 7u) * 2u;
}

// V consecutive 16-bit values (V = 1, 2 or 4) as one register-sized word.
template <int V>
struct Vec;
template <>
struct Vec<1> {
    using T = uint16_t;
};
template <>
struct Vec<2> {
    using T = uint32_t;
};
template <>
struct Vec<4> {
    using T = uint2;
};

template <int V>
__device__ __forceinline__ typename Vec<V>::T vzero()
{
    if constexpr (V == 4)
        return make_uint2(0u, 0u);
    else
        return typename Vec<V>::T(0);
}

template <bool F16, bool C_VEC, int V, bool ASYNC>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_any_kernel(const Params p)
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

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], kProducerThreads);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbarrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int M = p.M, N = p.N, K = p.K;
    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (N + BN - 1) / BN;
    const int ntiles = tiles_m * tiles_n;
    const int kblocks = (K + BK - 1) / BK;
    const uint64_t limit = p.limit_ns;

    if (warp < kProducerWarps) {
      if constexpr (ASYNC) {
        // ------------------------------------------------ producers (cp.async)
        // V = 2 or 4 (4- or 8-byte copies straight into the swizzled layout,
        // zero-filled outside M, N, K). A thread's copies for a K-slice form
        // one cp.async group; up to kAsyncDepth slices are in flight per
        // thread, and a slice is announced on full[] once the thread's own
        // copies of it have landed and been fenced for the tensor core, so
        // no registers hold operands and several slices stream at once.
        constexpr int A_ROW = BK / V, A_PER = BM * A_ROW / kProducerThreads;
        constexpr int A_STEP = kProducerThreads / A_ROW;
        constexpr int B_ROW = BN / V, B_PER = BK * B_ROW / kProducerThreads;
        constexpr int B_STEP = kProducerThreads / B_ROW;
        constexpr uint32_t VB = 2 * V;  // bytes per copy
        static_assert(kAsyncDepth < STAGES, "a reused stage must have been announced");
        const int tid = threadIdx.x;  // 0 .. 255 among the producer warps
        const int ar = tid / A_ROW, ac = (tid % A_ROW) * V;
        const int br = tid / B_ROW, bc = (tid % B_ROW) * V;
        uint32_t stage = 0, phase = 0, pending = 0, oldest = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok && !*abort; t += gridDim.x) {
            int m0, n0;
            tile_coords(t, tiles_m, tiles_n, m0, n0);
            const uint16_t *pa0 = p.A + (size_t)(m0 + ar) * K + ac;
            const uint16_t *pb0 = p.B + (size_t)br * N + (n0 + bc);
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1, limit, abort)) {
                    give_up(p.err, abort);
                    ok = false;
                    break;
                }
                const int k0 = kb * BK;
                const uint32_t sA = smem_u32(smem + stage * STAGE_BYTES);
                const uint32_t sB = sA + A_STAGE_BYTES;
    #pragma unroll
                for (int j = 0; j < A_PER; ++j) {
                    const int row = ar + j * A_STEP;
                    const bool in = m0 + row < M && k0 + ac < K;  // K % V == 0: all or none
                    const uint16_t *src = in ? pa0 + (size_t)j * A_STEP * K + k0 : p.A;
                    if constexpr (V == 4)
                        cp_async_8(sA + swz(row, ac), src, in ? VB : 0u);
                    else
                        cp_async_4(sA + swz(row, ac), src, in ? VB : 0u);
                }
    #pragma unroll 8
                for (int j = 0; j < B_PER; ++j) {
                    const int krow = br + j * B_STEP;
                    const bool in = k0 + krow < K && n0 + bc < N;  // N % V == 0
                    const uint16_t *src = in ? pb0 + (size_t)(k0 + j * B_STEP) * N : p.B;
                    const uint32_t dst = sB + (bc >> 6) * B_ATOM_BYTES + swz(krow, bc & 63);
                    if constexpr (V == 4)
                        cp_async_8(dst, src, in ? VB : 0u);
                    else
                        cp_async_4(dst, src, in ? VB : 0u);
                }
                cp_async_commit();
                if (++pending == kAsyncDepth) {
                    cp_async_wait<kAsyncDepth - 1>();  // the oldest slice has landed
                    fence_proxy_async_shared();
                    mbar_arrive(&full[oldest]);
                    oldest = oldest + 1 == STAGES ? 0 : oldest + 1;
                    --pending;
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // Announce the slices still in flight; on every path (including a
        // give-up) every copy lands before this thread goes on.
        cp_async_wait<0>();
        fence_proxy_async_shared();
        for (; pending > 0; --pending) {
            mbar_arrive(&full[oldest]);
            oldest = oldest + 1 == STAGES ? 0 : oldest + 1;
        }
      } else {
        // ------------------------------------------------ producers (plain loads)
        uint32_t stage = 0, phase = 0;
        for (int t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
            int m0, n0;
            tile_coords(t, tiles_m, tiles_n, m0, n0);
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1, limit, abort)) {
                    give_up(p.err, abort);
                    ok = false;
                    break;
                }
                const int k0 = kb * BK;
                uint8_t *sA = smem + stage * STAGE_BYTES;
                uint8_t *sB = sA + A_STAGE_BYTES;
                if constexpr (V == 1) {
                    // All of this lane's loads for the slice are issued before any
                    // store, so the slice costs one round trip to L2, not dozens.
                    // A: 128 rows x 64 k; warp w fills rows 16w .. 16w+15, lanes run along k.
                    // B: 64 k-rows x 256 n in four 64-column atoms; warp w fills k-rows
                    // 8w .. 8w+7, lanes run along n.
                    constexpr int AR = BM / kProducerWarps, AE = BK / 32;
                    constexpr int BR = BK / kProducerWarps, BE = BN / 32;
                    uint16_t va[AR][AE], vb[BR][BE];
    #pragma unroll
                    for (int rr = 0; rr < AR; ++rr) {
                        const int gm = m0 + warp * AR + rr;
    #pragma unroll
                        for (int e = 0; e < AE; ++e) {
                            const int gk = k0 + e * 32 + lane;
                            va[rr][e] =
                                (gm < M && gk < K) ? __ldg(p.A + (size_t)gm * K + gk) : (uint16_t)0;
                        }
                    }
    #pragma unroll
                    for (int kr = 0; kr < BR; ++kr) {
                        const int gk = k0 + warp * BR + kr;
    #pragma unroll
                        for (int e = 0; e < BE; ++e) {
                            const int gn = n0 + e * 32 + lane;
                            vb[kr][e] =
                                (gk < K && gn < N) ? __ldg(p.B + (size_t)gk * N + gn) : (uint16_t)0;
                        }
                    }
    #pragma unroll
                    for (int rr = 0; rr < AR; ++rr)
    #pragma unroll
                        for (int e = 0; e < AE; ++e)
                            *reinterpret_cast<uint16_t *>(sA + swz(warp * AR + rr, e * 32 + lane)) =
                                va[rr][e];
    #pragma unroll
                    for (int kr = 0; kr < BR; ++kr)
    #pragma unroll
                        for (int e = 0; e < BE; ++e) {
                            const int n = e * 32 + lane;
                            *reinterpret_cast<uint16_t *>(sB + (n >> 6) * B_ATOM_BYTES +
                                                          swz(warp * BR + kr, n & 63)) = vb[kr][e];
                        }
                } else {
                    // The same with V values per access: consecutive producer
                    // threads take consecutive vectors along a row; a thread's
                    // vectors share one column and step down the rows by a fixed
                    // stride, so one base pointer per operand serves all.
                    using W = typename Vec<V>::T;
                    constexpr int A_ROW = BK / V, A_PER = BM * A_ROW / kProducerThreads;
                    constexpr int A_STEP = kProducerThreads / A_ROW;  // rows between a thread's vectors
                    constexpr int B_ROW = BN / V, B_PER = BK * B_ROW / kProducerThreads;
                    constexpr int B_STEP = kProducerThreads / B_ROW;
                    const int tid = threadIdx.x;  // 0 .. 255 among the producer warps
                    const int ar = tid / A_ROW, ac = (tid % A_ROW) * V;
                    const int br = tid / B_ROW, bc = (tid % B_ROW) * V;
                    const int gka = k0 + ac, gnb = n0 + bc;
                    const uint16_t *pa = p.A + (size_t)(m0 + ar) * K + gka;
                    const uint16_t *pb = p.B + (size_t)(k0 + br) * N + gnb;
                    W va[A_PER], vb[B_PER];
    #pragma unroll
                    for (int j = 0; j < A_PER; ++j) {
                        const bool in = m0 + ar + j * A_STEP < M && gka < K;
                        va[j] = in ? __ldg(reinterpret_cast<const W *>(pa + (size_t)j * A_STEP * K))
                                   : vzero<V>();
                    }
    #pragma unroll
                    for (int j = 0; j < B_PER; ++j) {
                        const bool in = k0 + br + j * B_STEP < K && gnb < N;
                        vb[j] = in ? __ldg(reinterpret_cast<const W *>(pb + (size_t)j * B_STEP * N))
                                   : vzero<V>();
                    }
    #pragma unroll
                    for (int j = 0; j < A_PER; ++j)
                        *reinterpret_cast<W *>(sA + swz(ar + j * A_STEP, ac)) = va[j];
    #pragma unroll
                    for (int j = 0; j < B_PER; ++j)
                        *reinterpret_cast<W *>(sB + (bc >> 6) * B_ATOM_BYTES + swz(br + j * B_STEP, bc & 63)) =
                            vb[j];
                }
                fence_proxy_async_shared();
                mbar_arrive(&full[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok)
                break;
        }
      }
    } else if (warp == kMmaWarp) {
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
                        const uint64_t adesc = sdesc_sw128(sa + kk * UMMA_K * 2, 16, 1024);
                        const uint64_t bdesc =
                            sdesc_sw128(sb + kk * UMMA_K * 128, B_ATOM_BYTES, 1024);
                        umma_f16(d_tmem, adesc, bdesc, idesc<F16>(), (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued_any = true;
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok)
                    break;
                umma_commit(&tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            if (issued_any) {
                umma_commit(drain);
                volatile int no_abort = 0;
                mbar_wait_bounded(drain, 0, limit, &no_abort);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 9..12)
        const int quarter = warp & 3;
        uint32_t acc = 0, acc_phase = 0;
        for (int t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
            int m0, n0;
            tile_coords(t, tiles_m, tiles_n, m0, n0);
            if (!mbar_wait_bounded(&tfull[acc], acc_phase, limit, abort)) {
                give_up(p.err, abort);
                break;
            }
            tc_fence_after();
            const int row = m0 + quarter * 32 + lane;
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
            float *crow = p.C + (size_t)row * N;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + c * 32, r);
                tmem_wait_ld();
                if (c == BN / 32 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&tempty[acc]);
                }
                if (row < M) {
                    const int col = n0 + c * 32;
                    if constexpr (C_VEC) {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            if (col + v * 4 < N) {  // N % 4 == 0: all four or none
                                float4 o;
                                o.x = __uint_as_float(r[v * 4 + 0]);
                                o.y = __uint_as_float(r[v * 4 + 1]);
                                o.z = __uint_as_float(r[v * 4 + 2]);
                                o.w = __uint_as_float(r[v * 4 + 3]);
                                *reinterpret_cast<float4 *>(crow + col + v * 4) = o;
                            }
                    } else {
#pragma unroll
                        for (int v = 0; v < 32; ++v)
                            if (col + v < N)
                                crow[col + v] = __uint_as_float(r[v]);
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
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <bool F16, bool C_VEC, int V, bool ASYNC = false>
static cudaError_t launch(const TcLaunch &L, cudaStream_t stream)
{
    auto kernel = gemm_tc_any_kernel<F16, C_VEC, V, ASYNC>;
    static std::atomic<uint64_t> done{0};  // per instantiation
    const cudaError_t e = set_smem_limit_once(kernel, (int)SMEM_BYTES, done);
    if (e != cudaSuccess)
        return e;
    const long long ntiles = (long long)((L.M + BM - 1) / BM) * ((L.N + BN - 1) / BN);
    const int grid = (int)(ntiles < L.sm_count ? ntiles : L.sm_count);
    Params p{L.M, L.N, L.K, L.A, L.B, L.C, L.err, (unsigned long long)L.wait_limit_ns};
    kernel<<<grid, kThreads, SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

template <bool F16, bool C_VEC>
static cudaError_t launch_v(const TcLaunch &L, int v, cudaStream_t stream)
{
    // 8-byte copies through cp.async (several K-slices in flight): 344 -> 529
    // TFLOP/s at 4096 x 4100 x 4100 on GB300. 4-byte copies stay register-staged:
    // with twice the copy instructions cp.async was faster only at 8192 x 8190 x
    // 8190 (331 -> 354) and slower below (2048 x 2050 x 2050: 239 -> 209).
    return v == 4 ? launch<F16, C_VEC, 4, true>(L, stream)
           : v == 2 ? launch<F16, C_VEC, 2>(L, stream)
                    : launch<F16, C_VEC, 1>(L, stream);
}

} // namespace tcany

cudaError_t launch_gemm_tc_any(const TcLaunch &L, cudaStream_t stream)
{
    using namespace tcany;
    const bool c_vec = (L.N % 4 == 0) && ((reinterpret_cast<uintptr_t>(L.C) & 15) == 0);
    // Widest access that keeps every row of A and B aligned to it.
    const uintptr_t a = reinterpret_cast<uintptr_t>(L.A), b = reinterpret_cast<uintptr_t>(L.B);
    int v = 4;
    while (v > 1 && (L.K % v != 0 || L.N % v != 0 || (a % (2 * v)) != 0 || (b % (2 * v)) != 0))
        v /= 2;
    if (L.f16)
        return c_vec ? launch_v<true, true>(L, v, stream) : launch_v<true, false>(L, v, stream);
    return c_vec ? launch_v<false, true>(L, v, stream) : launch_v<false, false>(L, v, stream);
}

} // namespace rtm
