// bf16 x bf16 (or fp16 x fp16) -> fp32 product C = A.B for short products
// (M <= 128) whose A or B rows do not start on 16-byte boundaries, computed as
// its transpose C^T = B^T.A^T with K split over a cluster; and, without the
// swap, for tall, narrow products on such rows.
//
// The tiling is the transposed kernel's of gemm_tc_t.cu ("寄存器Tiling跨架构
// 解析", section 6: the accumulator tile is whatever the matrix instruction
// computes, and which operand feeds which side is free). A CTA owns 128
// columns of C (the MMA's M) and MN rows (MN = 32, 64 or 128, the next size
// >= M), and one of S K-ranges: the S CTAs of a cluster sum their partial
// tiles through distributed shared memory in rank order. Each 64-deep K-slice
// stages 64 k-rows x 128 columns of B (two 64-column atoms, MN-major: the
// MMA's A operand) and MN rows x 64 k of A (K-major: the MMA's B operand).
// Nearly every staged byte is B, and B is read once, so the product is bound
// by how fast B reaches shared memory. Without the swap (SWAP = false) the
// same kernel serves tall, narrow products (M > 128, N <= 128, long K): A
// (128 rows x 64 k, K-major) fills the MMA's 128-row side and B (64 k-rows x
// MN = 64 or 128 columns, MN-major) its N side, as in gemm_tc_t.cu.
//
// The TMA producer thread is replaced by producer warps that copy the slice
// with 2-, 4- or 8-byte accesses (the widest V for which every row of A and B
// starts on a 2V-byte boundary) into the swizzled layouts above (16-byte
// chunk c of a 128-byte row r at chunk c ^ (r mod 8)), zeros outside M, N, K.
// With 4- and 8-byte accesses eight warps issue cp.async copies straight into
// a 4-stage ring and keep three slices in flight per thread; 2-byte values
// (which cp.async cannot copy) are loaded into registers by sixteen warps
// and stored after they arrive. On GB300 the copies measured faster than
// register staging with three slices per thread (16 x 8190 x 8190: 48.2 ->
// 41.6 us; 16 x 8188 x 8188: 55.0 -> 34.8 us); a deeper ring (6 stages), 16
// copying warps or two CTAs per SM gained nothing. The ring stays small
// because the copies in flight pass through L1, which gets what the
// shared-memory carve-out leaves.
//
// With the swap, columns of C are TMEM lanes and rows of C TMEM columns
// (without it, the reverse): with S = 1 four epilogue warps store the
// accumulator directly (with the swap, for each row of C the 32 lanes of a
// warp write 32 consecutive floats; without it, a thread writes 32
// consecutive floats of its row, as float4 where C rows are 16-byte
// aligned); with S > 1 each CTA writes its partial tile into its idle stage
// memory, CTA r of the cluster sums TMEM columns [r MN / S, (r + 1) MN / S)
// of the partials over the cluster in rank order 0, 1, .., S-1 and stores
// them, and a second cluster barrier keeps every partial alive until all
// have been read. The MMA sequence, the K-ranges and the order of the sums
// are those of the TMA-fed kernel of gemm_tc_t.cu, so both give the same bits
// on the same values. C rows need only 4-byte alignment.
//
// Every mbarrier wait is bounded in time; a warp that gives up records
// GEMM_ERR_TIMEOUT in the device error word and every thread still reaches
// the cluster barriers.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tc_any_common.cuh"

namespace rtm {
namespace tcany {
namespace tshort {

constexpr int BNT = 128;  // columns of C per CTA: the MMA's M
constexpr uint32_t BT_BYTES = BK * BNT * 2;  // 16 KB: 64 k-rows x 128 columns of B
constexpr int kEpilogueWarps = 4;
constexpr int threads_of(int pw) { return (pw + 1 + kEpilogueWarps) * 32; }

template <int MN, int STG>
struct Cfg {
    static constexpr int STAGES = STG;
    static constexpr uint32_t AT_BYTES = MN * BK * 2;  // 4, 8 or 16 KB of A per stage
    static constexpr uint32_t STAGE_BYTES = BT_BYTES + AT_BYTES;
    static constexpr uint32_t RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int PITCH = MN + 4;  // floats per row of a partial tile in shared memory
    static constexpr uint32_t PART_BYTES = BNT * PITCH * 4;
    static constexpr size_t SMEM_BYTES = RING_BYTES + 256 /*barriers*/ + 1024 /*align*/;
    static_assert(PART_BYTES <= RING_BYTES, "partial tile must fit the stage ring");
};

// kind::f16, D fp32, A and B both bf16 (1) or both fp16 (0); N = MN, M = 128.
// SWAP: the MMA's A (= B^T) MN-major, its B (= A^T) K-major; otherwise A
// K-major and B MN-major.
template <bool F16, int MN, bool SWAP>
__host__ __device__ constexpr uint32_t idesc_t()
{
    return (1u << 4) | ((F16 ? 0u : 1u) << 7) | ((F16 ? 0u : 1u) << 10) |
           ((SWAP ? 1u : 0u) << 15) | ((SWAP ? 0u : 1u) << 16) | ((uint32_t)(MN >> 3) << 17) |
           ((uint32_t)(BNT >> 4) << 24);
}

struct Params {
    int M, N, K;
    const uint16_t *A;
    const uint16_t *B;
    float *C;
    int *err;
    unsigned long long limit_ns;
    int splits;         // CTAs per cluster, each summing one K-range
    int mute_producer;  // failure-detection self-test: the producer warps load nothing
    int c_vec;          // C rows 16-byte aligned (float4 row stores without the swap)
};

// One K-slice of 2-byte values (V = 1) in a producer thread's registers:
// AROWS rows of A (k0 .. k0+63) and 64 k-rows of B (BCOLS columns from n0), a
// lane per element, coalesced along k for A and along n for B; warp w holds
// rows AR w .. AR w + AR - 1 of A and k-rows BR w .. BR w + BR - 1 of B. A and
// B check their bounds apart: B's columns are interior for all but the last
// column tile whatever M is.
template <int PT, int AROWS, int BCOLS>
struct Slice1 {
    static constexpr int PW = PT / 32;
    static constexpr int AR = AROWS / PW, AE = BK / 32;
    static constexpr int BR = BK / PW, BE = BCOLS / 32;
    static_assert(AR >= 1 && AR * PW == AROWS && BR * PW == BK && BE >= 1,
                  "whole rows per producer warp");
    uint16_t a[AR][AE], b[BR][BE];

    __device__ __forceinline__ void load(const Params &p, int tid, int m0, int n0, int k0)
    {
        const int warp = tid >> 5, lane = tid & 31;
        const uint16_t *pa = p.A + (size_t)(m0 + warp * AR) * p.K + (k0 + lane);
        const uint16_t *pb = p.B + (size_t)(k0 + warp * BR) * p.N + (n0 + lane);
        const bool k_in = k0 + BK <= p.K;
        if (k_in && n0 + BCOLS <= p.N) {
#pragma unroll
            for (int kr = 0; kr < BR; ++kr)
#pragma unroll
                for (int e = 0; e < BE; ++e)
                    b[kr][e] = __ldg(pb + (size_t)kr * p.N + e * 32);
        } else {
#pragma unroll
            for (int kr = 0; kr < BR; ++kr)
#pragma unroll
                for (int e = 0; e < BE; ++e)
                    b[kr][e] = (k0 + warp * BR + kr < p.K && n0 + e * 32 + lane < p.N)
                                   ? __ldg(pb + (size_t)kr * p.N + e * 32)
                                   : (uint16_t)0;
        }
#pragma unroll
        for (int rr = 0; rr < AR; ++rr)
#pragma unroll
            for (int e = 0; e < AE; ++e)
                a[rr][e] = (m0 + warp * AR + rr < p.M && k0 + e * 32 + lane < p.K)
                               ? __ldg(pa + (size_t)rr * p.K + e * 32)
                               : (uint16_t)0;
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
                *reinterpret_cast<uint16_t *>(sB + (n >> 6) * B_ATOM_BYTES +
                                              swz(warp * BR + kr, n & 63)) = b[kr][e];
            }
    }
};

// Producer warps: 8 issuing cp.async copies, 16 loading 2-byte values.
constexpr int producer_warps(int v) { return v == 1 ? 16 : 8; }
constexpr int kStages = 4;

// 2-byte slices a producer thread keeps in registers (a register per value):
// two of up to 20 values (MN = 32 with the swap), one above, within the 80
// registers a thread of a 672-thread CTA can have (two of 24 spill).
template <typename Slice>
constexpr int ring_depth_2byte()
{
    return Slice::AR * Slice::AE + Slice::BR * Slice::BE <= 20 ? 2 : 1;
}

template <int V>
__device__ __forceinline__ void cp_async_v(uint32_t dst, const void *src, uint32_t bytes)
{
    if constexpr (V == 4)
        cp_async_8(dst, src, bytes);
    else
        cp_async_4(dst, src, bytes);
}

// The copies of one producer thread for V = 2 or 4 values per copy:
// consecutive threads take consecutive vectors along a row, and a thread's
// vectors share one column and step A_STEP (B_STEP) rows down, A_STEP a
// multiple of 8 and B_STEP of 4, so a vector's swizzled offset is one of two
// per thread (every other vector of B has the first one's swizzle phase, the
// others that of row + 4).
template <int V, int PT, int AROWS, int BCOLS>
struct AsyncPlan {
    static constexpr int A_ROW = BK / V, A_PER = AROWS * A_ROW / PT, A_STEP = PT / A_ROW;
    static constexpr int B_ROW = BCOLS / V, B_PER = BK * B_ROW / PT, B_STEP = PT / B_ROW;
    static_assert(A_PER >= 1 && A_PER * PT == AROWS * A_ROW && B_PER >= 1 &&
                      B_PER * PT == BK * B_ROW,
                  "every producer thread copies whole vectors of both operands");
    static_assert(A_STEP % 8 == 0 && B_STEP % 4 == 0, "swizzle phase fixed per vector");
    // Byte offset of B vector j from the offsets of rows br and br + 4.
    static __device__ __forceinline__ uint32_t b_off(int j, uint32_t db0, uint32_t db1)
    {
        if constexpr (B_STEP % 8 == 0)
            return db0 + (uint32_t)(j * B_STEP * 128);
        else
            return ((j & 1) ? db1 : db0) + (uint32_t)((j >> 1) * 8 * 128);
    }
};

template <bool F16, int MN, int V, bool SWAP>
__global__ void __launch_bounds__(threads_of(producer_warps(V)), 1)
    gemm_tc_any_t_kernel(const Params p)
{
    using Cf = Cfg<MN, kStages>;
    constexpr int STAGES = Cf::STAGES;
    constexpr int PW = producer_warps(V);
    constexpr int PT = PW * 32;
    constexpr int kMmaWarp = PW;
    // The MMA's 128-row side (first in a stage) holds B^T with the swap, A
    // without; its N side (after it) A^T or B.
    constexpr int AROWS = SWAP ? MN : BNT, BCOLS = SWAP ? BNT : MN;
    constexpr uint32_t A_OFF = SWAP ? BT_BYTES : 0u, B_OFF = SWAP ? 0u : BT_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cf::RING_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *done = empty + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.splits;
    const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
    const int unit = blockIdx.x / S;
    int m0, n0;
    if constexpr (SWAP) {
        const int tiles_n = (p.N + BNT - 1) / BNT;
        n0 = (unit % tiles_n) * BNT;
        m0 = (unit / tiles_n) * MN;
    } else {
        const int tiles_m = (p.M + BNT - 1) / BNT;
        m0 = (unit % tiles_m) * BNT;
        n0 = (unit / tiles_m) * MN;
    }
    const int kblocks = (p.K + BK - 1) / BK;
    const int per = (kblocks + S - 1) / S;
    const int kb_begin = min(kblocks, (int)rank * per);
    const int kb_end = min(kblocks, kb_begin + per);
    const int nslices = kb_end - kb_begin;
    const uint64_t limit = p.limit_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], PT);  // every producer thread arrives
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *abort = 0;
        fence_mbarrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, MN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < PW) {
        // ------------------------------------------------ producers
        if (p.mute_producer || nslices == 0) {
            // nothing to stage (the self-test mutes the loads: every wait gives up)
        } else if constexpr (V > 1) {
            // V = 2 or 4: cp.async copies straight into the swizzled layout
            // (zero-filled outside M, N, K), a thread's copies for a slice one
            // group; STAGES - 1 slices in flight per thread, each announced on
            // full[] once the thread's own copies of it have landed and been
            // fenced for the tensor core. No registers hold operands, so the
            // ring depth, not the register file, sets the bytes in flight.
            using SV = AsyncPlan<V, PT, AROWS, BCOLS>;
            constexpr int DEPTH = STAGES - 1;
            constexpr uint32_t VB = 2 * V;
            const int tid = threadIdx.x;
            const int ar = tid / SV::A_ROW, ac = (tid % SV::A_ROW) * V;
            const int br = tid / SV::B_ROW, bc = (tid % SV::B_ROW) * V;
            const uint32_t da = swz(ar, ac);
            const uint32_t db0 = (bc >> 6) * B_ATOM_BYTES + swz(br, bc & 63);
            const uint32_t db1 = (bc >> 6) * B_ATOM_BYTES + swz(br + 4, bc & 63);
            const size_t sa = (size_t)SV::A_STEP * p.K, sb = (size_t)SV::B_STEP * p.N;
            uint32_t stage = 0, phase = 0, pending = 0, oldest = 0;
            for (int s = 0; s < nslices; ++s) {
                if (!warp_wait(&empty[stage], phase ^ 1, limit, abort)) {
                    give_up(p.err, abort);
                    break;
                }
                const int k0 = (kb_begin + s) * BK;
                const uint32_t sB = smem_u32(smem + stage * Cf::STAGE_BYTES) + B_OFF;
                const uint32_t sA = smem_u32(smem + stage * Cf::STAGE_BYTES) + A_OFF + da;
                const uint16_t *pa = p.A + (size_t)(m0 + ar) * p.K + (k0 + ac);
                const uint16_t *pb = p.B + (size_t)(k0 + br) * p.N + (n0 + bc);
                const bool k_in = k0 + BK <= p.K;
                if (k_in && n0 + BCOLS <= p.N) {
#pragma unroll
                    for (int j = 0; j < SV::B_PER; ++j)
                        cp_async_v<V>(sB + SV::b_off(j, db0, db1), pb + j * sb, VB);
                } else {
                    const bool nb = n0 + bc < p.N;
#pragma unroll
                    for (int j = 0; j < SV::B_PER; ++j) {
                        const bool in = nb && k0 + br + j * SV::B_STEP < p.K;
                        cp_async_v<V>(sB + SV::b_off(j, db0, db1), in ? pb + j * sb : p.B,
                                      in ? VB : 0u);
                    }
                }
                if (k_in && m0 + AROWS <= p.M) {
#pragma unroll
                    for (int j = 0; j < SV::A_PER; ++j)
                        cp_async_v<V>(sA + j * SV::A_STEP * 128, pa + j * sa, VB);
                } else {
                    const bool ka = k0 + ac < p.K;
#pragma unroll
                    for (int j = 0; j < SV::A_PER; ++j) {
                        const bool in = ka && m0 + ar + j * SV::A_STEP < p.M;
                        cp_async_v<V>(sA + j * SV::A_STEP * 128, in ? pa + j * sa : p.A,
                                      in ? VB : 0u);
                    }
                }
                cp_async_commit();
                if (++pending == DEPTH) {
                    cp_async_wait<DEPTH - 1>();  // the oldest slice has landed
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
            // Announce the slices still in flight; on every path (including a
            // give-up) every copy lands before this thread goes on.
            cp_async_wait<0>();
            fence_proxy_async_shared();
            for (; pending > 0; --pending) {
                mbar_arrive(&full[oldest]);
                oldest = oldest + 1 == STAGES ? 0 : oldest + 1;
            }
        } else {
            using Slice = Slice1<PT, AROWS, BCOLS>;
            constexpr int R = ring_depth_2byte<Slice>();
            const int tid = threadIdx.x;
            uint32_t stage = 0, phase = 0;
            int next = 0, left = nslices;
            auto load_next = [&](Slice &s) {
                if (next < nslices) {
                    s.load(p, tid, m0, n0, (kb_begin + next) * BK);
                    ++next;
                }
            };
            // Store the oldest slice loaded into the next stage and announce it;
            // false once every slice is out or a wait gave up.
            auto publish = [&](const Slice &cur) {
                if (!warp_wait(&empty[stage], phase ^ 1, limit, abort)) {
                    give_up(p.err, abort);
                    return false;
                }
                uint8_t *st = smem + stage * Cf::STAGE_BYTES;
                cur.store(st + A_OFF, st + B_OFF, tid);
                fence_proxy_async_shared();
                mbar_arrive(&full[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
                return --left > 0;
            };
            auto step = [&](const Slice &cur, Slice &fut) {
                load_next(fut);
                return publish(cur);
            };
            if constexpr (R == 1) {
                Slice s0;
                do
                    load_next(s0);
                while (publish(s0));
            } else {
                static_assert(R == 2, "one or two slices in registers");
                Slice s0, s1;
                load_next(s0);
                while (step(s0, s1) && step(s1, s0)) {
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool issued_any = false;
            for (int kb = kb_begin; kb < kb_end; ++kb) {
                if (!mbar_wait_bounded(&full[stage], phase, limit, abort)) {
                    give_up(p.err, abort);
                    break;
                }
                tc_fence_after();
                const uint32_t sbig = smem_u32(smem + stage * Cf::STAGE_BYTES);  // MMA's A
                const uint32_t ssmall = sbig + BT_BYTES;                           // MMA's B
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                    // MN-major side: 64-wide atoms B_ATOM_BYTES apart, 16 k-rows per step.
                    // K-major side: rows of 128 B, 8-row groups 1024 B apart, 32 B per step.
                    uint64_t adesc, bdesc;
                    if constexpr (SWAP) {
                        adesc = sdesc_sw128(sbig + kk * UMMA_K * 128, B_ATOM_BYTES, 1024);
                        bdesc = sdesc_sw128(ssmall + kk * UMMA_K * 2, 16, 1024);
                    } else {
                        adesc = sdesc_sw128(sbig + kk * UMMA_K * 2, 16, 1024);
                        bdesc = sdesc_sw128(ssmall + kk * UMMA_K * 128, B_ATOM_BYTES, 1024);
                    }
                    umma_f16(tmem_base, adesc, bdesc, idesc_t<F16, MN, SWAP>(),
                             (kb != kb_begin || kk != 0) ? 1u : 0u);
                }
                issued_any = true;
                umma_commit(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (issued_any) {
                umma_commit(done);
                volatile int no_abort = 0;
                mbar_wait_bounded(done, 0, limit, &no_abort);  // before TMEM is freed
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps PW+1 .. PW+4)
        const int quarter = warp & 3;         // the TMEM lanes this warp may read
        const int col = quarter * 32 + lane;  // TMEM lane: column n0 + col (swap) or row m0 + col of C
        const bool have = nslices > 0;
        bool ok = true;
        if (have && !mbar_wait_bounded(done, 0, limit, abort)) {
            give_up(p.err, abort);
            ok = false;
        }
        tc_fence_after();
        const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16);
        if (S == 1) {
            if (ok && have) {
#pragma unroll 1
                for (int c = 0; c < MN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + c * 32, r);
                    tmem_wait_ld();
                    if constexpr (SWAP) {
                        // for each row of C the warp's 32 lanes store 32 consecutive floats
                        const int gn = n0 + col;
                        const int rows = min(32, p.M - (m0 + c * 32));
                        if (gn < p.N) {
                            float *cp = p.C + (size_t)(m0 + c * 32) * p.N + gn;
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j < rows)
                                    cp[(size_t)j * p.N] = __uint_as_float(r[j]);
                        }
                    } else {
                        // a thread stores 32 consecutive floats of its row of C
                        const int gm = m0 + col;
                        const int gn0 = n0 + c * 32;
                        if (gm < p.M) {
                            float *cp = p.C + (size_t)gm * p.N + gn0;
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                if (p.c_vec && gn0 + 4 * v + 3 < p.N) {
                                    *reinterpret_cast<float4 *>(cp + 4 * v) = make_float4(
                                        __uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                        __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                                } else {
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        if (gn0 + 4 * v + e < p.N)
                                            cp[4 * v + e] = __uint_as_float(r[4 * v + e]);
                                }
                            }
                        }
                    }
                }
            }
        } else {
            float *part = reinterpret_cast<float *>(smem);
#pragma unroll 1
            for (int c = 0; c < MN / 32; ++c) {
                uint32_t r[32];
                if (have && ok) {
                    tmem_ld_32x32b_x32(t_row + c * 32, r);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        r[j] = 0u;  // an empty K-range contributes zeros
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<uint4 *>(part + col * Cf::PITCH + c * 32 + 4 * q) =
                        make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
            }
        }
    }

    if (S > 1) {
        cluster_sync();  // every partial tile of the cluster is in shared memory
        if (warp > kMmaWarp) {
            // TMEM lane `col` of every CTA: sum its columns [r MN / S, (r + 1) MN / S)
            const int col = (warp & 3) * 32 + lane;
            const int cols = MN / S;
            const int c0 = (int)rank * cols;
            const uint32_t mine = smem_u32(smem) + (uint32_t)(col * Cf::PITCH) * 4u;
            for (int cc = 0; cc < cols; cc += 4) {
                const uint32_t off = (uint32_t)(c0 + cc) * 4u;
                float4 acc = ld_shared_cluster_v4(mapa_shared(mine + off, 0));
                for (int q = 1; q < S; ++q) {
                    const float4 v = ld_shared_cluster_v4(mapa_shared(mine + off, (uint32_t)q));
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
                if constexpr (SWAP) {
                    const int gn = n0 + col, gm = m0 + c0 + cc;
                    if (gn < p.N) {
                        float *cp = p.C + (size_t)gm * p.N + gn;
                        if (gm + 0 < p.M) cp[0] = acc.x;
                        if (gm + 1 < p.M) cp[(size_t)p.N] = acc.y;
                        if (gm + 2 < p.M) cp[(size_t)2 * p.N] = acc.z;
                        if (gm + 3 < p.M) cp[(size_t)3 * p.N] = acc.w;
                    }
                } else {
                    const int gm = m0 + col, gn = n0 + c0 + cc;
                    if (gm < p.M) {
                        float *cp = p.C + (size_t)gm * p.N + gn;
                        if (p.c_vec && gn + 3 < p.N) {
                            *reinterpret_cast<float4 *>(cp) = acc;
                        } else {
                            if (gn + 0 < p.N) cp[0] = acc.x;
                            if (gn + 1 < p.N) cp[1] = acc.y;
                            if (gn + 2 < p.N) cp[2] = acc.z;
                            if (gn + 3 < p.N) cp[3] = acc.w;
                        }
                    }
                }
            }
        }
        cluster_sync();  // no CTA leaves while a peer may still read its partial
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, MN);
    }
}

template <bool F16, int MN, int V, bool SWAP>
static cudaError_t launch_mn(const TcLaunch &L, int splits, cudaStream_t stream)
{
    using Cf = Cfg<MN, kStages>;
    auto kernel = gemm_tc_any_t_kernel<F16, MN, V, SWAP>;
    constexpr int kThreadsT = threads_of(producer_warps(V));
    static std::atomic<uint64_t> done{0};  // per instantiation
    // The smallest carve-out that holds the ring (of the SM's 228 KB): the
    // producers' copies in flight pass through L1, which gets the rest.
    cudaError_t e = set_smem_limit_once(
        kernel, (int)Cf::SMEM_BYTES, done,
        (int)((Cf::SMEM_BYTES * 100 + 228 * 1024 - 1) / (228 * 1024)));
    if (e != cudaSuccess)
        return e;
    const long long tiles = SWAP ? (long long)((L.N + BNT - 1) / BNT) * ((L.M + MN - 1) / MN)
                                 : (long long)((L.M + BNT - 1) / BNT) * ((L.N + MN - 1) / MN);
    // Every tile's cluster resident at once: halve the split while more
    // clusters would be launched than fit.
    static std::atomic<int> resident[4][64] = {};  // clusters of 1, 2, 4, 8
    while (splits > 1) {
        const int slot = splits == 2 ? 1 : splits == 4 ? 2 : 3;
        const int fit = resident_clusters(kernel, splits, kThreadsT, Cf::SMEM_BYTES, resident[slot]);
        if (fit <= 0 || tiles <= fit)
            break;
        splits /= 2;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * splits), 1, 1);
    cfg.blockDim = dim3(kThreadsT, 1, 1);
    cfg.dynamicSmemBytes = Cf::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int c_vec = (L.N % 4 == 0) && ((reinterpret_cast<uintptr_t>(L.C) & 15) == 0);
    Params p{L.M, L.N, L.K, L.A, L.B, L.C, L.err, (unsigned long long)L.wait_limit_ns, splits,
             L.mute_producer, c_vec};
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <bool F16, int MN, bool SWAP>
static cudaError_t launch_v(const TcLaunch &L, int v, int splits, cudaStream_t stream)
{
    return v == 4 ? launch_mn<F16, MN, 4, SWAP>(L, splits, stream)
           : v == 2 ? launch_mn<F16, MN, 2, SWAP>(L, splits, stream)
                    : launch_mn<F16, MN, 1, SWAP>(L, splits, stream);
}

template <bool F16>
static cudaError_t launch_f(const TcLaunch &L, int v, int splits, bool swap, cudaStream_t stream)
{
    if (!swap)
        return tcs_cols(L.N) == 64 ? launch_v<F16, 64, false>(L, v, splits, stream)
                                   : launch_v<F16, 128, false>(L, v, splits, stream);
    const int mn = tct_rows(L.M);
    return mn == 32 ? launch_v<F16, 32, true>(L, v, splits, stream)
           : mn == 64 ? launch_v<F16, 64, true>(L, v, splits, stream)
                      : launch_v<F16, 128, true>(L, v, splits, stream);
}

} // namespace tshort
} // namespace tcany

cudaError_t launch_gemm_tc_any_t(const TcLaunch &L, int splits, bool swap, cudaStream_t stream)
{
    using namespace tcany;
    if ((swap ? L.M : L.N) > 128 || (splits != 1 && splits != 2 && splits != 4 && splits != 8))
        return cudaErrorInvalidValue;
    const int v = access_width(L);
    return L.f16 ? tshort::launch_f<true>(L, v, splits, swap, stream)
                 : tshort::launch_f<false>(L, v, splits, swap, stream);
}

} // namespace rtm
