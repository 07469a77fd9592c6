// Helpers shared by the TMA-fed SIMT fp32 kernels (sgemm_tma.cu,
// sgemm_tma_rect.cu): 16-byte shared-memory vector accesses, the L2-grouped
// tile raster, and the fp32 tensor maps the TMA loads read.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace rtm {
namespace simt_tma_common {

__device__ __forceinline__ float4 lds128(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, float x, float y, float z, float w)
{
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(x), "f"(y), "f"(z),
                 "f"(w)
                 : "memory");
}

// Tile `bid` of a tiles_m x tiles_n grid walked in groups of G tile-rows:
// inside a group the walk goes down the G rows of one tile-column before the
// next column, so the CTAs resident at once share A rows and B columns in L2.
template <int G>
__device__ __forceinline__ void grouped_tile(int bid, int tiles_m, int tiles_n, int &tile_m,
                                             int &tile_n)
{
    const int group_size = G * tiles_n;
    const int group = bid / group_size;
    const int first_m = group * G;
    const int rows = min(tiles_m - first_m, G);
    const int in_group = bid - group * group_size;
    tile_m = first_m + in_group % rows;
    tile_n = in_group / rows;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A rows x cols fp32 matrix, row-major with rows cols * 4 bytes apart, read in
// boxes of box_rows x box_cols; zeros outside the matrix.
inline bool encode_f32_map(EncodeTiledFn fn, CUtensorMap *map, const float *base, uint64_t rows,
                           uint64_t cols, uint32_t box_cols, uint32_t box_rows,
                           CUtensorMapSwizzle swizzle, uint64_t ld = 0)
{
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {(ld ? ld : cols) * 4};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

} // namespace simt_tma_common
} // namespace rtm
