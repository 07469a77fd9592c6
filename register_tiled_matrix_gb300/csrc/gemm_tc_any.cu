// bf16/fp16 -> fp32 product C = A.B on tcgen05 for M > 128 and any 2-byte
// aligned pointers: the path for rows that do not start on 16-byte
// boundaries (K % 8 != 0 or N % 8 != 0, or offset pointers), which the
// tensor-memory-access unit cannot address, when no workspace allows
// re-pitched copies. (Short products, M <= 128, take the transposed kernel of
// gemm_tc_any_t.cu.)
//
// The TMA producer of the CTA-pair kernel (gemm_tc2.cu) is replaced by
// producer warps that load the A and B slices and store them into the same
// 128-byte-swizzled shared-memory layouts the MMA descriptors describe
// (16-byte chunk c of a 128-byte row r at chunk c ^ (r mod 8)), writing zeros
// outside M, N, K. Each producer thread then makes its shared-memory writes
// visible to the tensor core (fence.proxy.async) and arrives on the stage's
// barrier. Loads and stores move V consecutive values at once (V = 1, 2 or 4:
// 2-, 4- or 8-byte accesses), the largest V for which every row of A and B
// starts on a 2V-byte boundary (K and N multiples of V, A and B 2V-byte
// aligned), so a vector never straddles a row end or a 16-byte swizzle chunk.
#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tc_any_common.cuh"

namespace rtm {
namespace tcany {

struct Params {
    int M, N, K;
    const uint16_t *A;
    const uint16_t *B;
    float *C;
    int *err;
    unsigned long long limit_ns;
    int mute_producer;  // failure-detection self-test: the producer warps load nothing
};

// ---------------------------------------------------------------- CTA pairs
// The producers on the two-SM form of tcgen05 (cta_group::2): a cluster of
// two CTAs computes a 256 x 256 C tile with one MMA stream issued by the even
// CTA, and each CTA's producer warps stage only its half of the operands —
// 128 rows of A and 128 columns of B per 64-deep K-slice, 32 KB instead of
// the 48 KB of a lone 128 x 256 tile — into its own shared memory. On GB300,
// 4- and 8-byte copies move at most about 36-39 bytes per clock per SM from L2
// into shared memory, where 16-byte cp.async moves 102: with these copies the
// bytes each SM must stage per tensor-core cycle bound the kernel, and the
// pair cuts them by a third. Loads in flight are staged in L1, which gets
// what the shared-memory carve-out leaves, so the ring is only four stages
// deep (146 KB) and the launch asks for the smallest carve-out that holds it.
// Rows 0-127 of a tile accumulate in the even CTA's tensor memory, rows
// 128-255 in the odd CTA's (two accumulators per CTA); each CTA's four
// epilogue warps store their rows through shared memory, 32 consecutive
// floats per store instruction.
//
// Every producer thread fences its shared-memory writes for the async proxy
// and arrives on its own CTA's full[] barrier. In the odd CTA one otherwise
// idle thread (lane 0 of the MMA warp) waits for
// each of its CTA's slices and forwards it with one cluster-scope release
// arrival on the even CTA's full[] barrier, where the MMA issuer waits for
// both CTAs. MMA completions are multicast to both CTAs' empty[] and
// accumulator barriers.
namespace pair {

constexpr int PM = 256;  // tile rows (128 per CTA)
constexpr int PN = 256;  // tile columns (128 staged per CTA)
constexpr int HM = 128;
constexpr int HN = 128;
// Producer warps per CTA (a template parameter PW of the kernel): 16 for the
// register-staged producers, whose loads in flight grow with the warps
// (8192 x 8190 x 8190: 8 warps 1.70 ms, 16 warps 1.51 ms), 8 for cp.async
// (8192 x 8188 x 8188: 1.38 ms against 1.43 ms with 16). Warp PW issues the
// MMAs (even CTA) or forwards slices (odd CTA); warps PW+1 .. PW+4 store C.
constexpr int pair_threads(int pw) { return (pw + 1 + 4) * 32; }
constexpr int PSTAGES = 4;
constexpr int kPairAsyncDepth = PSTAGES - 1;
constexpr int kGroupMPair = 8;
constexpr uint32_t PA_BYTES = HM * BK * 2;             // 16 KB
constexpr uint32_t PSTAGE_BYTES = PA_BYTES + BK * HN * 2;  // + two 64-column B atoms
constexpr uint32_t PTMEM_COLS = 2 * PN;
constexpr int kEpiPitch = 33;  // floats per row of an epilogue block
constexpr uint32_t EPI_WARP_BYTES = 32 * kEpiPitch * 4;
constexpr uint32_t OFF_BARS = PSTAGES * PSTAGE_BYTES;
constexpr uint32_t OFF_EPI = OFF_BARS + 256;
constexpr size_t PSMEM_BYTES = OFF_EPI + 4 * EPI_WARP_BYTES + 1024 /*align*/;
constexpr uint16_t kBothCtas = 0x3;
constexpr uint16_t kEvenCta = 0x1;

// kind::f16, D fp32, A K-major, B MN-major, N = 256, M = 256 (both CTAs).
template <bool F16>
__host__ __device__ constexpr uint32_t idesc_pair()
{
    return (1u << 4) | ((F16 ? 0u : 1u) << 7) | ((F16 ? 0u : 1u) << 10) | (0u << 15) |
           (1u << 16) | ((uint32_t)(PN >> 3) << 17) | ((uint32_t)(PM >> 4) << 24);
}

__device__ __forceinline__ void pair_tile_coords(int t, int tiles_m, int tiles_n, int &m0, int &n0)
{
    const int group_size = kGroupMPair * tiles_n;
    const int group = t / group_size;
    const int first_m = group * kGroupMPair;
    const int rows = min(tiles_m - first_m, kGroupMPair);
    const int in_group = t - group * group_size;
    m0 = (first_m + in_group % rows) * PM;
    n0 = (in_group / rows) * PN;
}

// One K-slice of this CTA's operands held in registers by a producer thread:
// V values per access (V = 2 or 4), consecutive threads on consecutive
// vectors along a row, a thread's vectors A_STEP (B_STEP) rows apart. A
// vector's place in the swizzled layout depends on its row only through
// row mod 8, which the steps fix at compile time: A_STEP is a multiple of 8,
// B_STEP of 4 (every other vector shares the first one's phase).
template <int V, int PT>
struct Staged {
    using W = typename Vec<V>::T;
    static constexpr int A_ROW = BK / V, A_PER = HM * A_ROW / PT;
    static constexpr int A_STEP = PT / A_ROW;
    static constexpr int B_ROW = HN / V, B_PER = BK * B_ROW / PT;
    static constexpr int B_STEP = PT / B_ROW;
    static_assert(A_STEP % 8 == 0 && B_STEP % 4 == 0, "swizzle phase fixed per vector");
    W a[A_PER], b[B_PER];

    // A rows r0.., columns k0..k0+63; B rows k0..k0+63, columns c0..c0+127;
    // zeros outside M, N, K (K % V == 0 and N % V == 0: a vector is all in or out).
    __device__ __forceinline__ void load(const Params &p, int tid, int r0, int c0, int k0)
    {
        const int ar = tid / A_ROW, ac = (tid % A_ROW) * V;
        const int br = tid / B_ROW, bc = (tid % B_ROW) * V;
        const uint16_t *pa = p.A + (size_t)(r0 + ar) * p.K + (k0 + ac);
        const uint16_t *pb = p.B + (size_t)(k0 + br) * p.N + (c0 + bc);
        const size_t sa = (size_t)A_STEP * p.K, sb = (size_t)B_STEP * p.N;
        if (r0 + HM <= p.M && c0 + HN <= p.N && k0 + BK <= p.K) {
#pragma unroll
            for (int j = 0; j < A_PER; ++j)
                a[j] = __ldg(reinterpret_cast<const W *>(pa + j * sa));
#pragma unroll
            for (int j = 0; j < B_PER; ++j)
                b[j] = __ldg(reinterpret_cast<const W *>(pb + j * sb));
        } else {
            const bool ka = k0 + ac < p.K, nb = c0 + bc < p.N;
#pragma unroll
            for (int j = 0; j < A_PER; ++j)
                a[j] = (ka && r0 + ar + j * A_STEP < p.M)
                           ? __ldg(reinterpret_cast<const W *>(pa + j * sa))
                           : vzero<V>();
#pragma unroll
            for (int j = 0; j < B_PER; ++j)
                b[j] = (nb && k0 + br + j * B_STEP < p.K)
                           ? __ldg(reinterpret_cast<const W *>(pb + j * sb))
                           : vzero<V>();
        }
    }

    __device__ __forceinline__ void store(uint8_t *sA, uint8_t *sB, int tid) const
    {
        const int ar = tid / A_ROW, ac = (tid % A_ROW) * V;
        const int br = tid / B_ROW, bc = (tid % B_ROW) * V;
        uint8_t *da = sA + swz(ar, ac);
        uint8_t *db = sB + (bc >> 6) * B_ATOM_BYTES;
        uint8_t *db0 = db + swz(br, bc & 63);
        uint8_t *db1 = db + swz(br + 4, bc & 63);
#pragma unroll
        for (int j = 0; j < A_PER; ++j)
            *reinterpret_cast<W *>(da + j * A_STEP * 128) = a[j];
#pragma unroll
        for (int j = 0; j < B_PER; ++j) {
            if constexpr (B_STEP % 8 == 0)
                *reinterpret_cast<W *>(db0 + j * B_STEP * 128) = b[j];
            else
                *reinterpret_cast<W *>(((j & 1) ? db1 : db0) + (j >> 1) * 8 * 128) = b[j];
        }
    }
};

// The same for 2-byte accesses (V = 1): lane per element, coalesced along k
// for A and along n for B; warp w holds rows AR w .. AR w + AR - 1 of A and
// k-rows BR w .. of B (AR a multiple of 8, so a row's swizzle phase is fixed).
template <int PT>
struct Staged1 {
    static constexpr int PW = PT / 32;
    static constexpr int AR = HM / PW, AE = BK / 32;
    static constexpr int BR = BK / PW, BE = HN / 32;
    static_assert(AR % 8 == 0, "swizzle phase fixed per row");
    uint16_t a[AR][AE], b[BR][BE];

    __device__ __forceinline__ void load(const Params &p, int tid, int r0, int c0, int k0)
    {
        const int warp = tid >> 5, lane = tid & 31;
        const uint16_t *pa = p.A + (size_t)(r0 + warp * AR) * p.K + (k0 + lane);
        const uint16_t *pb = p.B + (size_t)(k0 + warp * BR) * p.N + (c0 + lane);
        if (r0 + HM <= p.M && c0 + HN <= p.N && k0 + BK <= p.K) {
#pragma unroll
            for (int rr = 0; rr < AR; ++rr)
#pragma unroll
                for (int e = 0; e < AE; ++e)
                    a[rr][e] = __ldg(pa + (size_t)rr * p.K + e * 32);
#pragma unroll
            for (int kr = 0; kr < BR; ++kr)
#pragma unroll
                for (int e = 0; e < BE; ++e)
                    b[kr][e] = __ldg(pb + (size_t)kr * p.N + e * 32);
        } else {
#pragma unroll
            for (int rr = 0; rr < AR; ++rr)
#pragma unroll
                for (int e = 0; e < AE; ++e)
                    a[rr][e] = (r0 + warp * AR + rr < p.M && k0 + e * 32 + lane < p.K)
                                   ? __ldg(pa + (size_t)rr * p.K + e * 32)
                                   : (uint16_t)0;
#pragma unroll
            for (int kr = 0; kr < BR; ++kr)
#pragma unroll
                for (int e = 0; e < BE; ++e)
                    b[kr][e] = (k0 + warp * BR + kr < p.K && c0 + e * 32 + lane < p.N)
                                   ? __ldg(pb + (size_t)kr * p.N + e * 32)
                                   : (uint16_t)0;
        }
    }

    __device__ __forceinline__ void store(uint8_t *sA, uint8_t *sB, int tid) const
    {
        const int warp = tid >> 5, lane = tid & 31;
#pragma unroll
        for (int rr = 0; rr < AR; ++rr)
#pragma unroll
            for (int e = 0; e < AE; ++e)
                *reinterpret_cast<uint16_t *>(sA + swz(warp * AR + rr, e * 32 + lane)) = a[rr][e];
#pragma unroll
        for (int kr = 0; kr < BR; ++kr)
#pragma unroll
            for (int e = 0; e < BE; ++e) {
                const int n = e * 32 + lane;
                *reinterpret_cast<uint16_t *>(sB + (n >> 6) * B_ATOM_BYTES + swz(warp * BR + kr, n & 63)) =
                    b[kr][e];
            }
    }
};

template <bool F16, int V, bool ASYNC, int PW>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads(PW), 1)
    gemm_tc_any_pair_kernel(const Params p)
{
    constexpr int kPairProducerWarps = PW;
    constexpr int kPairProducerThreads = PW * 32;
    constexpr int kPairMmaWarp = PW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    uint64_t *empty = full + PSTAGES;
    uint64_t *tfull = empty + PSTAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: the even CTA, which issues the MMAs
    const bool even = rank == 0;
    const int cluster_id = blockIdx.x >> 1;
    const int num_clusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            // this CTA's producer threads; in the even CTA also the odd CTA's forwarder
            mbar_init(&full[s], kPairProducerThreads + (even ? 1 : 0));
            mbar_init(&empty[s], 1);                  // one multicast commit per stage use
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);  // even CTA: the pair's eight epilogue warps
        }
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbarrier_init();
    }
    if (warp == kPairMmaWarp) {
        tmem_alloc_pair(tmem_slot, PTMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int M = p.M, N = p.N, K = p.K;
    const int tiles_m = (M + PM - 1) / PM;
    const int tiles_n = (N + PN - 1) / PN;
    const int ntiles = tiles_m * tiles_n;
    const int kblocks = (K + BK - 1) / BK;
    const uint64_t limit = p.limit_ns;

    if (warp < kPairProducerWarps) {
        // ------------------------------------------------ producers (both CTAs)
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        if (p.mute_producer) {
            // failure-detection self-test: nothing arrives on full[], every wait gives up
        } else if constexpr (ASYNC) {
            // V = 4: 8-byte cp.async straight into the swizzled layout, zero-
            // filled outside M, N, K; kPairAsyncDepth slices in flight per thread,
            // a slice announced once the warp's copies of it have landed.
            constexpr int A_ROW = BK / V, A_PER = HM * A_ROW / kPairProducerThreads;
            constexpr int A_STEP = kPairProducerThreads / A_ROW;
            constexpr int B_ROW = HN / V, B_PER = BK * B_ROW / kPairProducerThreads;
            constexpr int B_STEP = kPairProducerThreads / B_ROW;
            static_assert(kPairAsyncDepth < PSTAGES, "a reused stage must have been announced");
            const int tid = threadIdx.x;
            const int ar = tid / A_ROW, ac = (tid % A_ROW) * V;
            const int br = tid / B_ROW, bc = (tid % B_ROW) * V;
            static_assert(A_STEP % 8 == 0 && B_STEP % 8 == 0, "swizzle phase fixed per vector");
            const uint32_t da = swz(ar, ac);
            const uint32_t db = (bc >> 6) * B_ATOM_BYTES + swz(br, bc & 63);
            const size_t sa = (size_t)A_STEP * K, sb = (size_t)B_STEP * N;
            uint32_t pending = 0, oldest = 0;
            for (int t = cluster_id; t < ntiles && ok; t += num_clusters) {
                int m0, n0;
                pair_tile_coords(t, tiles_m, tiles_n, m0, n0);
                const int r0 = m0 + (int)rank * HM, c0 = n0 + (int)rank * HN;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!warp_wait(&empty[stage], phase ^ 1, limit, abort)) {
                        give_up(p.err, abort);
                        ok = false;
                        break;
                    }
                    const int k0 = kb * BK;
                    const uint32_t sA = smem_u32(smem + stage * PSTAGE_BYTES) + da;
                    const uint32_t sB = smem_u32(smem + stage * PSTAGE_BYTES) + PA_BYTES + db;
                    const uint16_t *pa = p.A + (size_t)(r0 + ar) * K + (k0 + ac);
                    const uint16_t *pb = p.B + (size_t)(k0 + br) * N + (c0 + bc);
                    if (r0 + HM <= M && c0 + HN <= N && k0 + BK <= K) {
#pragma unroll
                        for (int j = 0; j < A_PER; ++j)
                            cp_async_8(sA + j * A_STEP * 128, pa + j * sa, 8u);
#pragma unroll
                        for (int j = 0; j < B_PER; ++j)
                            cp_async_8(sB + j * B_STEP * 128, pb + j * sb, 8u);
                    } else {
                        // zero-filled outside M, N, K (K % V == 0, N % V == 0)
                        const bool ka = k0 + ac < K, nb = c0 + bc < N;
#pragma unroll
                        for (int j = 0; j < A_PER; ++j) {
                            const bool in = ka && r0 + ar + j * A_STEP < M;
                            cp_async_8(sA + j * A_STEP * 128, in ? pa + j * sa : p.A, in ? 8u : 0u);
                        }
#pragma unroll
                        for (int j = 0; j < B_PER; ++j) {
                            const bool in = nb && k0 + br + j * B_STEP < K;
                            cp_async_8(sB + j * B_STEP * 128, in ? pb + j * sb : p.B, in ? 8u : 0u);
                        }
                    }
                    cp_async_commit();
                    if (++pending == kPairAsyncDepth) {
                        cp_async_wait<kPairAsyncDepth - 1>();  // the oldest slice has landed
                        fence_proxy_async_shared();
                        mbar_arrive(&full[oldest]);
                        oldest = oldest + 1 == PSTAGES ? 0 : oldest + 1;
                        --pending;
                    }
                    if (++stage == PSTAGES) {
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
                oldest = oldest + 1 == PSTAGES ? 0 : oldest + 1;
            }
        } else {
            // V = 1 or 2: register-staged. For V = 2 a ring of three slices per
            // thread: the loads of the slice two ahead (possibly of a later tile)
            // are issued before this slice is stored, so a warp keeps three
            // slices' loads in flight. A 2-byte slice takes twice the registers:
            // two in flight spill (240 bytes) under the 80 registers a thread of
            // this 672-thread CTA can have, so V = 1 keeps one.
            const int tid = threadIdx.x;
            using Slice = std::conditional_t<V == 1, Staged1<kPairProducerThreads>,
                                             Staged<V, kPairProducerThreads>>;
            int lt = cluster_id, lkb = 0, lr0 = 0, lc0 = 0;  // next slice to load
            auto origin = [&](int t) {
                int m0, n0;
                pair_tile_coords(t, tiles_m, tiles_n, m0, n0);
                lr0 = m0 + (int)rank * HM;
                lc0 = n0 + (int)rank * HN;
            };
            auto load_next = [&](Slice &buf) {
                if (lt >= ntiles)
                    return;
                buf.load(p, tid, lr0, lc0, lkb * BK);
                if (++lkb == kblocks) {
                    lkb = 0;
                    lt += num_clusters;
                    if (lt < ntiles)
                        origin(lt);
                }
            };
            // the grid has at most one cluster per tile: this CTA owns a tile
            long long remaining =
                (long long)((ntiles - 1 - cluster_id) / num_clusters + 1) * kblocks;
            origin(lt);
            // Store `cur` (the oldest slice loaded) into the next stage and announce it.
            auto publish = [&](Slice &cur) {
                if (!warp_wait(&empty[stage], phase ^ 1, limit, abort)) {
                    give_up(p.err, abort);
                    return false;
                }
                uint8_t *sA = smem + stage * PSTAGE_BYTES;
                cur.store(sA, sA + PA_BYTES, tid);
                fence_proxy_async_shared();
                mbar_arrive(&full[stage]);
                if (++stage == PSTAGES) {
                    stage = 0;
                    phase ^= 1;
                }
                return --remaining > 0;
            };
            if constexpr (V == 1) {
                Slice s0;
                do
                    load_next(s0);
                while (publish(s0));
            } else {
                // load the slice two ahead into `fut`, then publish `cur`
                auto step = [&](Slice &cur, Slice &fut) {
                    load_next(fut);
                    return publish(cur);
                };
                Slice s0, s1, s2;
                load_next(s0);
                load_next(s1);
                while (step(s0, s2) && step(s1, s0) && step(s2, s1)) {
                }
            }
        }
    } else if (warp == kPairMmaWarp) {
        // ------------------------------------------------ MMA issuer (even CTA), forwarder (odd)
        if (even && lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool issued_any = false;
            for (int t = cluster_id; t < ntiles && !*abort; t += num_clusters) {
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, limit, abort)) {
                    give_up(p.err, abort);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * PN;
                bool ok = true;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, limit, abort)) {
                        give_up(p.err, abort);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * PSTAGE_BYTES);
                    const uint32_t sb = sa + PA_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint64_t adesc = sdesc_sw128(sa + kk * UMMA_K * 2, 16, 1024);
                        const uint64_t bdesc =
                            sdesc_sw128(sb + kk * UMMA_K * 128, B_ATOM_BYTES, 1024);
                        umma_f16_pair(d_tmem, adesc, bdesc, idesc_pair<F16>(),
                                      (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued_any = true;
                    umma_commit_pair_multicast(&empty[stage], kBothCtas);
                    if (++stage == PSTAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok)
                    break;
                umma_commit_pair_multicast(&tfull[acc], kBothCtas);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            if (issued_any) {
                umma_commit_pair_multicast(drain, kEvenCta);
                volatile int no_abort = 0;
                mbar_wait_bounded(drain, 0, limit, &no_abort);
            }
        } else if (!even && lane == 0) {
            // Forwarder: this CTA's slices, in order, to the even CTA's full[].
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int t = cluster_id; t < ntiles && ok; t += num_clusters)
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, limit, abort)) {
                        give_up(p.err, abort);
                        ok = false;
                        break;
                    }
                    mbar_arrive_cluster(mapa_shared(smem_u32(&full[stage]), 0));
                    if (++stage == PSTAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (both CTAs)
        // Lane i holds row i of a 32 x 32 block: written to shared memory as
        // row i (pitch 33 floats: 32 lanes, 32 banks), read back by columns so
        // that lane j stores column j of each row.
        const int quarter = warp & 3;
        float *blk = reinterpret_cast<float *>(smem + OFF_EPI + quarter * EPI_WARP_BYTES);
        uint32_t acc = 0, acc_phase = 0;
        for (int t = cluster_id; t < ntiles; t += num_clusters) {
            int m0, n0;
            pair_tile_coords(t, tiles_m, tiles_n, m0, n0);
            if (!warp_wait(&tfull[acc], acc_phase, limit, abort)) {
                give_up(p.err, abort);
                break;
            }
            tc_fence_after();
            const int row0 = m0 + (int)rank * HM + quarter * 32;
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * PN;
            const int rows = min(32, M - row0);
#pragma unroll 1
            for (int c = 0; c < PN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + c * 32, r);
                tmem_wait_ld();
                if (c == PN / 32 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_cluster_tmem_free(mapa_shared(smem_u32(&tempty[acc]), 0));
                }
#pragma unroll
                for (int v = 0; v < 32; ++v)
                    blk[lane * kEpiPitch + v] = __uint_as_float(r[v]);
                __syncwarp();
                const int col = n0 + c * 32 + lane;
                if (col < N) {
                    float *cp = p.C + (size_t)row0 * N + col;
#pragma unroll 4
                    for (int rr = 0; rr < rows; ++rr)
                        cp[(size_t)rr * N] = blk[rr * kEpiPitch + lane];
                }
                __syncwarp();
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still signal or read it
    if (warp == kPairMmaWarp) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, PTMEM_COLS);
    }
}

template <bool F16, int V, bool ASYNC, int PW>
static cudaError_t launch_pair(const TcLaunch &L, cudaStream_t stream)
{
    auto kernel = gemm_tc_any_pair_kernel<F16, V, ASYNC, PW>;
    constexpr int kPairThreads = pair_threads(PW);
    static std::atomic<uint64_t> done{0};  // per instantiation
    // The smallest carve-out that holds the ring (of the SM's 228 KB): the
    // producers' loads in flight are staged in L1, which gets the rest.
    // 8192 x 8190 x 8190 with 6 stages and no hint 2.17 ms, 4 stages 1.80 ms,
    // 4 stages and this hint 1.70 ms.
    cudaError_t e = set_smem_limit_once(kernel, (int)PSMEM_BYTES, done,
                                        (int)((PSMEM_BYTES * 100 + 228 * 1024 - 1) / (228 * 1024)));
    if (e != cudaSuccess)
        return e;
    // Pairs resident at once (the persistent grid), per device; 0: not yet known.
    static std::atomic<int> max_clusters[64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    int clusters_max = (dev >= 0 && dev < 64) ? max_clusters[dev].load() : 0;
    if (clusters_max <= 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (L.sm_count / 2), 1, 1);
        cfg.blockDim = dim3(kPairThreads, 1, 1);
        cfg.dynamicSmemBytes = PSMEM_BYTES;
        if (cudaOccupancyMaxActiveClusters(&clusters_max, kernel, &cfg) != cudaSuccess ||
            clusters_max <= 0) {
            cudaGetLastError();
            clusters_max = L.sm_count / 2;
        }
        if (dev >= 0 && dev < 64)
            max_clusters[dev].store(clusters_max);
    }
    const long long ntiles = (long long)((L.M + PM - 1) / PM) * ((L.N + PN - 1) / PN);
    const int clusters = (int)(ntiles < clusters_max ? ntiles : clusters_max);
    Params p{L.M, L.N, L.K, L.A, L.B, L.C, L.err, (unsigned long long)L.wait_limit_ns,
             L.mute_producer};
    kernel<<<2 * clusters, kPairThreads, PSMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

} // namespace pair

} // namespace tcany

cudaError_t launch_gemm_tc_any_pair(const TcLaunch &L, cudaStream_t stream)
{
    using namespace tcany;
    const int v = access_width(L);
    if (L.f16)
        return v == 4 ? pair::launch_pair<true, 4, true, 8>(L, stream)
               : v == 2 ? pair::launch_pair<true, 2, false, 16>(L, stream)
                        : pair::launch_pair<true, 1, false, 16>(L, stream);
    return v == 4 ? pair::launch_pair<false, 4, true, 8>(L, stream)
           : v == 2 ? pair::launch_pair<false, 2, false, 16>(L, stream)
                    : pair::launch_pair<false, 1, false, 16>(L, stream);
}

} // namespace rtm
