// Pieces shared by the tensor-core kernels whose producer warps load A and B
// with plain 2-, 4- or 8-byte accesses and store them into the 128-byte-
// swizzled shared-memory layouts the MMA descriptors describe: the path for
// rows that do not start on 16-byte boundaries, which the tensor-memory-
// access unit cannot address (gemm_tc_any.cu: 128 x 256 tiles and CTA pairs;
// gemm_tc_any_t.cu: short products computed as their transpose).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace rtm {
namespace tcany {

constexpr int BK = 64;      // 64 16-bit values = one 128-byte swizzle row
constexpr int UMMA_K = 16;  // K of one kind::f16 MMA
constexpr uint32_t B_ATOM_BYTES = BK * 64 * 2;  // 64 k-rows x 64 columns, MN-major

// Shared-memory matrix descriptor, 128-byte swizzle (SM100 layout type 2).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
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

// A bounded wait whose outcome every lane of the warp shares: true only when
// the phase completed for all lanes and no warp has given up. Producer and
// epilogue warps synchronise inside their loops, so no lane may leave a loop
// that the others stay in.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t limit,
                                          volatile int *abort)
{
    const bool got = mbar_wait_bounded(bar, parity, limit, abort);
    return __all_sync(0xffffffffu, got && !*abort);
}

// Widest access (values) that keeps every row of A and B aligned to it: K and
// N multiples of V, A and B 2V-byte aligned, so a vector never straddles a row
// end or a 16-byte swizzle chunk.
inline int access_width(const TcLaunch &L)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(L.A), b = reinterpret_cast<uintptr_t>(L.B);
    int v = 4;
    while (v > 1 && (L.K % v != 0 || L.N % v != 0 || (a % (2 * v)) != 0 || (b % (2 * v)) != 0))
        v /= 2;
    return v;
}

} // namespace tcany
} // namespace rtm
