// Row re-pitching copy for the TMA-fed kernels: moves a row-major matrix of
// 2-byte (or, as pairs of them, 4-byte) values whose rows do not start on
// 16-byte boundaries (an odd number
// of columns modulo 8, or an offset base pointer) into a buffer whose rows do,
// so the tensor-memory-access unit can stage it. This is the global level of
// the pages' tiling made possible on Blackwell: a TMA box must start on a
// 16-byte boundary, a plain row-major operand need not.
//
// One thread writes one 16-byte chunk (8 values) of a destination row. It
// reads the one or two 16-byte-aligned source chunks that hold those 8
// values and shifts them into place in registers; it never reads a 16-byte
// chunk that holds no byte of the source matrix, so no read leaves the pages
// the source occupies. Memory-bound: each source byte is read about once from
// DRAM (the second chunk is the next thread's first) and each destination
// byte written once.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"

namespace rtm {
namespace pack {

// Bytes s .. s+15 of the 32-byte window (lo, hi); s is even, 0 .. 14.
__device__ __forceinline__ uint4 window16(const uint4 lo, const uint4 hi, uint32_t s)
{
    const uint32_t w0 = lo.x, w1 = lo.y, w2 = lo.z, w3 = lo.w;
    const uint32_t w4 = hi.x, w5 = hi.y, w6 = hi.z, w7 = hi.w;
    const bool by8 = (s & 8u) != 0, by4 = (s & 4u) != 0;
    // Whole-word shift by (s >> 2) in two selection steps.
    const uint32_t v0 = by8 ? w2 : w0, v1 = by8 ? w3 : w1, v2 = by8 ? w4 : w2;
    const uint32_t v3 = by8 ? w5 : w3, v4 = by8 ? w6 : w4, v5 = by8 ? w7 : w5;
    const uint32_t u0 = by4 ? v1 : v0, u1 = by4 ? v2 : v1, u2 = by4 ? v3 : v2;
    const uint32_t u3 = by4 ? v4 : v3, u4 = by4 ? v5 : v4;
    uint4 o;
    if (s & 2u) {  // half-word shift: high half of one word, low half of the next
        o.x = __funnelshift_r(u0, u1, 16);
        o.y = __funnelshift_r(u1, u2, 16);
        o.z = __funnelshift_r(u2, u3, 16);
        o.w = __funnelshift_r(u3, u4, 16);
    } else {
        o = make_uint4(u0, u1, u2, u3);
    }
    return o;
}

template <typename Index>
__global__ void __launch_bounds__(256) pack_rows_kernel(const uint16_t *__restrict__ src,
                                                        Index rows, Index cols,
                                                        uint16_t *__restrict__ dst, Index ld)
{
    const Index chunks_per_row = (cols + 7) / 8;
    const Index total = rows * chunks_per_row;
    const uintptr_t src_end = reinterpret_cast<uintptr_t>(src) + (uintptr_t)rows * cols * 2;
    const Index stride = (Index)gridDim.x * blockDim.x;
    for (Index i = (Index)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const Index r = i / chunks_per_row;
        const Index c = i - r * chunks_per_row;
        const uintptr_t a = reinterpret_cast<uintptr_t>(src + (size_t)r * cols + (size_t)c * 8);
        const uintptr_t a0 = a & ~uintptr_t(15);
        const uint32_t s = (uint32_t)(a - a0);
        // The chunk at a0 holds the first value; the next one is needed only
        // when the 8 values straddle two chunks, and is read only if it holds
        // a byte of the matrix (values past the row end land in the padding).
        const uint4 lo = __ldg(reinterpret_cast<const uint4 *>(a0));
        uint4 hi = make_uint4(0u, 0u, 0u, 0u);
        if (s != 0 && a0 + 16 < src_end)
            hi = __ldg(reinterpret_cast<const uint4 *>(a0 + 16));
        *reinterpret_cast<uint4 *>(dst + (size_t)r * ld + (size_t)c * 8) = window16(lo, hi, s);
    }
}

} // namespace pack

cudaError_t launch_pack_rows_2b(const uint16_t *src, int64_t rows, int64_t cols, uint16_t *dst,
                                int64_t ld, int sm_count, cudaStream_t stream)
{
    if (rows <= 0 || cols <= 0)
        return cudaSuccess;
    const int64_t total = rows * ((cols + 7) / 8);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)sm_count * 8;  // 8 resident 256-thread blocks per SM
    if (blocks > cap)
        blocks = cap;
    if (total + (int64_t)blocks * 256 < ((int64_t)1 << 31) && ld < ((int64_t)1 << 31))
        pack::pack_rows_kernel<int32_t><<<(unsigned)blocks, 256, 0, stream>>>(
            src, (int32_t)rows, (int32_t)cols, dst, (int32_t)ld);
    else
        pack::pack_rows_kernel<int64_t><<<(unsigned)blocks, 256, 0, stream>>>(src, rows, cols,
                                                                               dst, ld);
    return cudaGetLastError();
}

// A row of cols 4-byte values is a row of 2 cols 2-byte values, and a stride
// of ld (a multiple of 4) one of 2 ld (a multiple of 8): the same copy.
cudaError_t launch_pack_rows_4b(const float *src, int64_t rows, int64_t cols, float *dst,
                                int64_t ld, int sm_count, cudaStream_t stream)
{
    return launch_pack_rows_2b(reinterpret_cast<const uint16_t *>(src), rows, 2 * cols,
                               reinterpret_cast<uint16_t *>(dst), 2 * ld, sm_count, stream);
}

} // namespace rtm
